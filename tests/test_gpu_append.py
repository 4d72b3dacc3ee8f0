"""Decode-time append on the GPU against the oracle.

New KV entries join each request's host-resident history (blog commentary, opening;
paper abstract: the full KV history lives in host memory); appends are interleaved
with resolutions, some at positions that are resident (rewrites), some not, some
skipped, and everything -- tables, outputs, slot bytes and the host store's bytes --
must equal the oracle's.
"""
import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen
from oracle import Oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,B", [("tiny", 1), ("dsa", 4), ("quest", 2)])
def test_append_interleaved_with_resolutions(name, B):
    hs.build()
    tracegen.build()
    w = tracegen.WORKLOADS[name]
    T = 12
    ctx = hs.Context(B, w.C, w.S, w.E)
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w, B=B)
    host_ref = ctx.host_kv().copy()  # the oracle's own copy of the history
    sel = tracegen.trace(w, T=T, B=B)
    sd = torch.from_numpy(sel).cuda()
    o = Oracle(B, w.C, w.S, w.E)
    rng = np.random.default_rng(7)
    out = torch.empty_like(sd[0])
    miss = torch.empty(B, dtype=torch.int32, device="cuda")
    for t in range(T):
        ctx.resolve(sd[t], out, miss)
        o_out, o_miss, _ = o.resolve(host_ref, ctx.host_stride, sel[t])
        assert np.array_equal(out.cpu().numpy(), o_out) and np.array_equal(miss.cpu().numpy(), o_miss), t
        # new entries: a resident position (rewrite), a fresh one, or none
        pos = np.empty(B, dtype=np.int32)
        for b in range(B):
            r = rng.integers(3)
            pos[b] = sel[t, b, rng.integers(w.k)] if r == 0 else (rng.integers(w.C) if r == 1 else -1)
        rows = rng.integers(0, 256, size=(B, w.E), dtype=np.uint8)
        ctx.append(torch.from_numpy(rows).cuda(), torch.from_numpy(pos).cuda())
        assert o.append(host_ref, pos, rows) == 0
    torch.cuda.synchronize()
    assert np.array_equal(ctx.host_kv(), host_ref)
    assert np.array_equal(ctx.device_kv().cpu().numpy(), o.dev)
    for name_, ref in (("page_table", o.pt), ("slot_token", o.tok), ("last_use", o.lu), ("step", o.t)):
        assert np.array_equal(getattr(ctx, name_)().cpu().numpy(), ref), name_
    # out of range: reported, skipped
    ctx.clear_status()
    bad = torch.full((B,), w.C, dtype=torch.int32, device="cuda")
    ctx.append(torch.zeros((B, w.E), dtype=torch.uint8, device="cuda"), bad)
    assert ctx.status() == hs.HS_STATUS_RANGE
    assert np.array_equal(ctx.host_kv(), host_ref)
    ctx.close()
