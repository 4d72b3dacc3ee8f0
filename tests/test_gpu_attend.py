"""The consumer on the GPU: sparse MLA-style attention over the resolved slots, against
the oracle's fp64 attention.

Tolerance, from the kernel's arithmetic: the products are exact in fp32 and accumulate in
fp32; the softmax weights are computed with the hardware base-2 exponential (relative
error below 2^-21) and rounded to bf16 (relative error at most 2^-9) before the value
product, and the sum that normalises them adds the same rounded weights. A weight
perturbed by a relative e moves a convex combination by at most 2e times the weighted
magnitude of the values, so |o - o_ref| <= 2 * (2^-9 + eps_s) * sum_j w_j |V_jd|, where
eps_s covers the score rounding: at most 2^-9 * sm_scale * sum_d |q_d latent_jd| when the
latent is multiplied by a non-unit scale and rounded to bf16 (computed per head from the
data), and far below 2^-9 otherwise (scale 1: the decoded latent is exact; the fp32 sums
of 576 exact products). The test allows (2^-7 + 2 eps_s) times the oracle's weighted
magnitude plus 1e-5 for o, and for lse (natural-log units, where the same weight errors
move ln of the sum by at most 2^-8 + eps_s) 2^-7 + 2 eps_s + 1e-5 |lse|.
"""
import math

import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen
from oracle import Oracle

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -7


@pytest.fixture(scope="module", autouse=True)
def _built():
    hs.build()
    tracegen.build()
    import oracle
    oracle.build()


def bf16_tensor(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def run_attend(ctx, q, out_slots, sm_scale):
    B, H, _ = q.shape
    o = torch.full((B, H, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = ctx.attend_workspace(B, H, out_slots.shape[1])
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    ctx.attend(q, out_slots, o, lse, sm_scale, workspace=ws)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    return o.cpu().numpy(), lse.cpu().numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, absw, what, ds=None):
    """ds: per-head bound on the score change from rounding the scaled latent (None: 0)."""
    ds = np.zeros(o_ref.shape[0]) if ds is None else ds
    tol_o = (TOL + 2 * ds[:, None]) * absw + 1e-5
    bad = np.abs(o_gpu - o_ref) > tol_o
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs out of tolerance, worst "
                           f"{float(np.max(np.abs(o_gpu - o_ref) - tol_o))}")
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), ~fin), what
    tol_l = TOL + 2 * ds + 1e-5 * np.abs(np.where(fin, lse_ref, 0))
    assert (np.abs(lse_gpu[fin] - lse_ref[fin]) <= tol_l[fin]).all(), what


def gaussian_rows(n: int, seed: int, scale_lo: float = 0.25, scale_hi: float = 4.0) -> np.ndarray:
    """n entries with N(0,1) latent codes (E4M3 by PyTorch's rounding), random block scales
    and N(0,1) bf16 rotary values."""
    rng = np.random.default_rng(seed)
    rows = np.zeros((n, 656), dtype=np.uint8)
    codes = torch.from_numpy(rng.standard_normal((n, 512)).astype(np.float32)).to(torch.float8_e4m3fn)
    rows[:, :512] = codes.view(torch.uint8).numpy()
    rows[:, 512:528] = rng.uniform(scale_lo, scale_hi, size=(n, 4)).astype(np.float32).view(np.uint8).reshape(n, 16)
    rows[:, 528:] = bf16_tensor(rng.standard_normal((n, 64))).view(torch.int16).numpy().view(np.uint8).reshape(n, 128)
    return rows


def score_rounding(rows: np.ndarray, slots: np.ndarray, q_bits: np.ndarray, sm: float) -> np.ndarray:
    """Per head, max over the valid selections of 2^-9 sm sum_d |q_d| |latent_jd|: the score
    change when the scaled latent is rounded to bf16 (rows indexed by slot)."""
    used = rows[slots[slots >= 0]]
    lat = torch.from_numpy(used[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(used[:, 512:528].copy()).view(torch.float32).to(torch.float64).repeat_interleave(128, 1)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64)[:, :512]
    return (2.0 ** -9 * sm * (q.abs() @ (lat * sc).abs().T)).max(dim=1).values.numpy()


def resolved_context(w, T, B):
    """A context after T resolution steps of the trace: (ctx, selections, last out_slots)."""
    ctx = hs.Context(B, w.C, w.S, w.E)
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w, B=B)
    sel = tracegen.trace(w, T=T, B=B)
    sd = torch.from_numpy(sel).cuda()
    out = torch.empty((T, B, sel.shape[2]), dtype=torch.int32, device="cuda")
    miss = torch.empty((T, B), dtype=torch.int32, device="cuda")
    for t in range(T):
        ctx.resolve(sd[t], out[t], miss[t])
    torch.cuda.synchronize()
    return ctx, sel, out[T - 1]


@pytest.mark.parametrize("B,k,H,S", [
    (2, 512, 128, 1024),   # several key splits per request
    (3, 200, 64, 256),     # ragged last block, fewer heads
    (80, 96, 16, 128),     # one split per request (B x 2 CTAs >= SMs)
    (1, 33, 1, 64),        # one head, one key past a block
    (1, 5000, 32, 6000),   # more selections than one CTA stages: at least three key splits
])
def test_attend_matches_oracle_after_resolution(B, k, H, S):
    w = tracegen.Workload("att", 11, B=B, L=1, C=4 * S, S=S, k=k, E=656, kv_kind=tracegen.KV_DSA656,
                          T=6, keep_pct=70, zipf_s=1.1, seed=B * 7 + k)
    ctx, sel, out = resolved_context(w, w.T, B)
    rng = np.random.default_rng(k)
    q = bf16_tensor(rng.standard_normal((B, H, 576)))
    sm = 1.0 / math.sqrt(576)
    o_gpu, lse_gpu = run_attend(ctx, q.cuda(), out, sm)
    # the oracle resolves the same trace on its own and attends over its own slots
    host = ctx.host_kv()
    orc = Oracle(B, w.C, w.S, w.E)
    for t in range(w.T):
        o_out, _, _ = orc.resolve(host, ctx.host_stride, sel[t])
    assert np.array_equal(o_out, out.cpu().numpy())
    qb = q.view(torch.int16).numpy().view(np.uint16)
    for b in range(B):
        o_ref, lse_ref, absw = orc.attend(b, qb[b], o_out[b], sm)
        compare(o_gpu[b], lse_gpu[b], o_ref, lse_ref, absw, f"request {b}")
    ctx.close()


def _context_with_rows(rows_per_req, S):
    """Context whose slots 0..n-1 of request b hold rows_per_req[b] (one cold resolution)."""
    B = len(rows_per_req)
    n = max(len(r) for r in rows_per_req)
    C = max(n, 2)
    ctx = hs.Context(B, C, S, 656)
    host = ctx.host_kv()
    host[:] = 0
    for b, r in enumerate(rows_per_req):
        host[b, :len(r), :656] = r
    sel = np.full((B, n), -1, dtype=np.int32)
    for b, r in enumerate(rows_per_req):
        sel[b, :len(r)] = np.arange(len(r))
    out = torch.empty((B, n), dtype=torch.int32, device="cuda")
    miss = torch.empty(B, dtype=torch.int32, device="cuda")
    ctx.resolve(torch.from_numpy(sel).cuda(), out, miss)
    torch.cuda.synchronize()
    orc = Oracle(B, C, S, 656)
    o_out, _, _ = orc.resolve(host, ctx.host_stride, sel)
    return ctx, orc, out, o_out


def test_attend_non_unit_scales_and_padding():
    """Random block scales (the latent is rounded to bf16 after scaling), padded selections."""
    rows = [gaussian_rows(150, 1), gaussian_rows(97, 2)]
    ctx, orc, out, o_out = _context_with_rows(rows, S=160)
    rng = np.random.default_rng(3)
    out_np = out.cpu().numpy()
    out_np[0, ::7] = -1  # padding among the selections
    out_np[1, 90:] = -1  # and a padded tail
    o_out[0, ::7] = -1
    o_out[1, 90:] = -1
    H = 128
    q = bf16_tensor(rng.standard_normal((2, H, 576)) * 0.5)
    sm = 1.0 / math.sqrt(576)
    o_gpu, lse_gpu = run_attend(ctx, q.cuda(), torch.from_numpy(out_np).cuda(), sm)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    dev = ctx.device_kv().cpu().numpy()
    for b in range(2):
        o_ref, lse_ref, absw = orc.attend(b, qb[b], o_out[b], sm)
        ds = score_rounding(dev[b], o_out[b], qb[b], sm)
        compare(o_gpu[b], lse_gpu[b], o_ref, lse_ref, absw, f"scaled request {b}", ds)
    ctx.close()


def test_attend_rescales_when_scores_keep_growing():
    """Scores that grow by far more than 2^8 per 32-key block force the running maximum to
    move (and O in tensor memory to be rescaled) at every block."""
    n = 256
    rows = np.zeros((n, 656), dtype=np.uint8)
    rows[:, :512] = 0x38  # every latent code 1.0
    scales = (np.arange(1, n + 1) / 512.0).astype(np.float32)  # exact in bf16
    rows[:, 512:528] = np.repeat(scales[:, None], 4, axis=1).view(np.uint8)
    ctx, orc, out, o_out = _context_with_rows([rows], S=n)
    q = bf16_tensor(np.ones((1, 8, 576)))
    sm = 0.5
    o_gpu, lse_gpu = run_attend(ctx, q.cuda(), out, sm)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    o_ref, lse_ref, absw = orc.attend(0, qb[0], o_out[0], sm)
    compare(o_gpu[0], lse_gpu[0], o_ref, lse_ref, absw, "growing scores")
    ctx.close()


def test_attend_all_padding_and_permutation():
    rows = [gaussian_rows(64, 4)]
    ctx, orc, out, o_out = _context_with_rows(rows, S=64)
    rng = np.random.default_rng(5)
    q = bf16_tensor(rng.standard_normal((1, 32, 576))).cuda()
    o0, l0 = run_attend(ctx, q, torch.full((1, 64), -1, dtype=torch.int32, device="cuda"), 0.05)
    assert (o0 == 0).all() and np.isneginf(l0).all()
    # any order of the selections: the running maximum then moves at other blocks, so the
    # bf16 rounding of the weights differs, but both stay within the bound of the oracle
    perm = np.random.default_rng(6).permutation(64)
    qb = q.cpu().view(torch.int16).numpy().view(np.uint16)
    o_ref, lse_ref, absw = orc.attend(0, qb[0], o_out[0], 0.05)
    dev = ctx.device_kv().cpu().numpy()
    ds = score_rounding(dev[0], o_out[0], qb[0], 0.05)
    for order in (np.arange(64), perm, perm[::-1].copy()):
        a, la = run_attend(ctx, q, out[:, torch.from_numpy(order).cuda()].contiguous(), 0.05)
        compare(a[0], la[0], o_ref, lse_ref, absw, "reordered", ds)
    ctx.close()


def test_attend_negative_scale():
    """A negative softmax scale: the block maximum is then taken over the scaled scores key
    by key (the raw maximum is the scaled minimum), with and without padding."""
    rows = [gaussian_rows(300, 7), gaussian_rows(40, 8)]
    ctx, orc, out, o_out = _context_with_rows(rows, S=320)
    out_np = out.cpu().numpy()
    out_np[1, 33:] = -1
    o_out[1, 33:] = -1
    rng = np.random.default_rng(9)
    q = bf16_tensor(rng.standard_normal((2, 64, 576)))
    sm = -1.0 / math.sqrt(576)
    o_gpu, lse_gpu = run_attend(ctx, q.cuda(), torch.from_numpy(out_np).cuda(), sm)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    dev = ctx.device_kv().cpu().numpy()
    for b in range(2):
        o_ref, lse_ref, absw = orc.attend(b, qb[b], o_out[b], sm)
        ds = score_rounding(dev[b], o_out[b], qb[b], abs(sm))
        compare(o_gpu[b], lse_gpu[b], o_ref, lse_ref, absw, f"negative scale, request {b}", ds)
    ctx.close()


def test_attend_random_shapes():
    """Seeded random shapes: ragged last blocks, one to several key splits, any head count
    and padding scattered through the selections, so that every fill role (producers,
    softmax warps, rotary copies) meets partial blocks and missing keys. Two requests of
    each shape are checked against the oracle."""
    rng = np.random.default_rng(2027)
    for case in range(4):
        B = int(rng.integers(1, 41))
        k = int(rng.integers(1, 2601))
        S = k + int(rng.integers(0, 400))
        H = int(rng.choice([8, 40, 128]))
        w = tracegen.Workload("attr", 17, B=B, L=1, C=4 * S, S=S, k=k, E=656, kv_kind=tracegen.KV_DSA656,
                              T=3, keep_pct=60, zipf_s=1.1, seed=100 + case)
        ctx, sel, out = resolved_context(w, w.T, B)
        orc = Oracle(B, w.C, w.S, w.E)
        host = ctx.host_kv()
        for t in range(w.T):
            o_out, _, _ = orc.resolve(host, ctx.host_stride, sel[t])
        assert np.array_equal(o_out, out.cpu().numpy()), case
        pad = rng.random(o_out.shape) < 0.05  # padding among the selections
        o_out = np.where(pad, -1, o_out).astype(np.int32)
        q = bf16_tensor(rng.standard_normal((B, H, 576)))
        sm = 1.0 / math.sqrt(576)
        o_gpu, lse_gpu = run_attend(ctx, q.cuda(), torch.from_numpy(o_out).cuda(), sm)
        qb = q.view(torch.int16).numpy().view(np.uint16)
        for b in sorted({0, B - 1}):
            o_ref, lse_ref, absw = orc.attend(b, qb[b], o_out[b], sm)
            compare(o_gpu[b], lse_gpu[b], o_ref, lse_ref, absw, f"case {case} (B={B} k={k} S={S} H={H}) request {b}")
        ctx.close()


def test_attend_full_size_dsa_sampled():
    """32 requests x k = 2048 x 128 heads (the DSA workload), three requests checked."""
    w = tracegen.WORKLOADS["dsa"]
    T = 4
    ctx, sel, out = resolved_context(w, T, w.B)
    rng = np.random.default_rng(8)
    q = bf16_tensor(rng.standard_normal((w.B, 128, 576)))
    sm = 1.0 / math.sqrt(576)
    o_gpu, lse_gpu = run_attend(ctx, q.cuda(), out, sm)
    host = ctx.host_kv()
    out_np = out.cpu().numpy()
    qb = q.view(torch.int16).numpy().view(np.uint16)
    C, E = w.C, w.E
    row_bytes = C * ctx.host_stride
    for b in (0, 17, 31):
        orc = Oracle(1, C, w.S, E)
        for t in range(T):
            o_out, _, _ = orc.resolve_request(0, ctx.host_kv_address() + b * row_bytes, ctx.host_stride, sel[t, b])
        assert np.array_equal(o_out, out_np[b])
        o_ref, lse_ref, absw = orc.attend(0, qb[b], o_out, sm)
        compare(o_gpu[b], lse_gpu[b], o_ref, lse_ref, absw, f"dsa request {b}")
    ctx.close()


def test_attend_in_a_cuda_graph_equals_eager():
    """hs_attend is enqueue-only: captured in a graph and replayed, it gives the eager result."""
    w = tracegen.Workload("attg", 13, B=4, L=1, C=2048, S=512, k=384, E=656, kv_kind=tracegen.KV_DSA656,
                          T=3, keep_pct=70, zipf_s=1.1, seed=5)
    ctx, sel, out = resolved_context(w, w.T, w.B)
    H = 128
    q = bf16_tensor(np.random.default_rng(2).standard_normal((w.B, H, 576))).cuda()
    nbytes = ctx.attend_workspace(w.B, H, w.k)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    o_e = torch.empty((w.B, H, 512), device="cuda")
    l_e = torch.empty((w.B, H), device="cuda")
    ctx.attend(q, out, o_e, l_e, 0.05, workspace=ws)
    o_g = torch.zeros_like(o_e)
    l_g = torch.zeros_like(l_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ctx.attend(q, out, o_g, l_g, 0.05, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o_e, o_g) and torch.equal(l_e, l_g)
    assert ctx.status() == 0
    ctx.close()


def test_attend_rejects_bad_calls():
    ctx = hs.Context(2, 64, 32, 656)
    q = torch.zeros((2, 8, 576), dtype=torch.bfloat16, device="cuda")
    sl = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    o = torch.empty((2, 8, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(hs.HsError):
        ctx.attend(torch.zeros((2, 129, 576), dtype=torch.bfloat16, device="cuda"), sl,
                   torch.empty((2, 129, 512), device="cuda"), torch.empty((2, 129), device="cuda"), 0.1)
    with pytest.raises(hs.HsError):
        ctx.attend(q[:1], sl[:1], o[:1], lse[:1], 0.1)
    ctx.close()
    other = hs.Context(2, 64, 32, 64)
    with pytest.raises(hs.HsError):
        other.attend(q, sl, o, lse, 0.1)
    other.close()
