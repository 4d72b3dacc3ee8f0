"""Pins for the oracle's consumer: sparse MLA-style attention over the resolved slots.

Sources of truth other than the oracle itself:
  * the OCP E4M3 format: fixed code values from its definition, and all 256 codes
    against PyTorch's float8_e4m3fn conversion (a library routine);
  * the definition of softmax attention evaluated by library routines (torch's fp64
    softmax, matmul and logsumexp) on small random cases;
  * closed forms: one valid selection (o = V, lse = s), k copies of one entry
    (o = V, lse = s + ln k), no valid selection (o = 0, lse = -inf), and invariance
    under reordering the selections.
"""
import math

import numpy as np
import pytest
import torch

E = 656


def dsa_rows(n: int, seed: int) -> np.ndarray:
    """n random 656-byte entries: finite e4m3 codes, scales in [0.25, 4), bf16 rope."""
    rng = np.random.default_rng(seed)
    rows = np.zeros((n, E), dtype=np.uint8)
    codes = rng.integers(0, 0x7F, size=(n, 512), dtype=np.uint8)  # 0x00..0x7E: finite
    codes |= (rng.integers(0, 2, size=(n, 512)) << 7).astype(np.uint8)
    rows[:, :512] = codes
    rows[:, 512:528] = rng.uniform(0.25, 4.0, size=(n, 4)).astype(np.float32).view(np.uint8).reshape(n, 16)
    rope = torch.from_numpy(rng.standard_normal((n, 64)).astype(np.float32)).to(torch.bfloat16)
    rows[:, 528:] = rope.view(torch.int16).numpy().view(np.uint8).reshape(n, 128)
    return rows


def bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def library_attention(rows: np.ndarray, q_bits: np.ndarray, sm_scale: float):
    """Reference by library routines: torch's e4m3 and bf16 conversions, fp64 softmax."""
    t = torch.from_numpy(rows)
    lat = t[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    sc = t[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    lat = lat * sc.repeat_interleave(128, dim=1)
    rope = t[:, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
    K = torch.cat([lat, rope], dim=1)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    s = sm_scale * (q @ K.T)
    return (torch.softmax(s, dim=1) @ lat).numpy(), torch.logsumexp(s, dim=1).numpy()


def _resolved(Oracle, rows_per_req, S, lib_path=None):
    """An oracle state whose slots hold the given entries (resolved from a host store)."""
    R, C = len(rows_per_req), max(len(r) for r in rows_per_req)
    host = np.zeros((R, C, E), dtype=np.uint8)
    for b, r in enumerate(rows_per_req):
        host[b, :len(r)] = r
    o = Oracle(R, C, S, E, lib_path=lib_path)
    sel = np.full((R, C), -1, dtype=np.int32)
    for b, r in enumerate(rows_per_req):
        sel[b, :len(r)] = np.arange(len(r))
    out, _, _ = o.resolve(host, E, sel)
    return o, host, out


def run_attend(Oracle, lib_path=None):
    rng = np.random.default_rng(5)
    # library reference on small random cases (with padding among the selections)
    for seed, (H, n) in enumerate([(3, 6), (1, 1), (5, 9)]):
        rows = dsa_rows(n, seed)
        o, host, out = _resolved(Oracle, [rows], S=max(n, 2), lib_path=lib_path)
        q = bf16_bits(rng.standard_normal((H, 576)))
        slots = out[0, :n].copy()
        keep = np.ones(n, dtype=bool)
        if n > 2:
            slots[1] = -1
            keep[1] = False
        sm = 1.0 / math.sqrt(576)
        got, lse, absw = o.attend(0, q, slots, sm)
        ref_o, ref_lse = library_attention(rows[keep], q, sm)
        assert np.allclose(got, ref_o, rtol=1e-11, atol=1e-12)
        assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
        assert (absw >= np.abs(got) - 1e-12).all()
    # closed forms
    rows = dsa_rows(3, 9)
    o, host, out = _resolved(Oracle, [rows], S=4, lib_path=lib_path)
    q = bf16_bits(rng.standard_normal((2, 576)))
    V, _ = library_attention(rows[:1], q, 0.1)
    got, lse, _ = o.attend(0, q, out[0, :1], 0.1)  # one entry
    assert np.allclose(got, V, rtol=1e-13, atol=0) and np.isfinite(lse).all()
    got4, lse4, _ = o.attend(0, q, np.repeat(out[0, :1], 4), 0.1)  # four copies of it
    assert np.allclose(got4, V, rtol=1e-13, atol=1e-15) and np.allclose(lse4, lse + math.log(4), rtol=0, atol=1e-12)
    got0, lse0, _ = o.attend(0, q, np.full(5, -1, dtype=np.int32), 0.1)  # nothing valid
    assert (got0 == 0).all() and np.isneginf(lse0).all()
    perm = o.attend(0, q, out[0, [2, 0, 1]], 0.1)
    base = o.attend(0, q, out[0, :3], 0.1)
    assert np.allclose(perm[0], base[0], rtol=1e-13, atol=1e-14) and np.allclose(perm[1], base[1], atol=1e-13)


def test_attention_pins(oracle_mod):
    run_attend(oracle_mod.Oracle)


def test_e4m3_codes(oracle_mod):
    """Fixed points of the E4M3 definition, and all 256 codes against PyTorch's decoder."""
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
             0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for c, v in fixed.items():
        assert oracle_mod.e4m3(c) == v, hex(c)
    assert math.isnan(oracle_mod.e4m3(0x7F)) and math.isnan(oracle_mod.e4m3(0xFF))
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle_mod.e4m3(c) for c in range(256)])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])
