"""The allocation-free entry point gives the same results as hs_resolve.

hs_resolve_noalloc exists for callers that cannot call cudaMalloc -- engines whose pool
allocator owns all GPU memory, or set-up code running while a stream is captured into a
CUDA graph. They pass every buffer themselves; the library's only scratch is a fixed
device array inside the library. This test plays such a caller: it owns the state
buffers (torch allocations standing in for the caller's pool) and checks, call after
call, that the results are identical to the context-based entry point on the same
inputs. Everything compared is integers or bytes, so equality is exact.

The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen

pytestmark = pytest.mark.gpu


def _noalloc(lib, w, host_addr, stride, st, sel, out, miss, status):
    return lib.hs_resolve_noalloc(torch.cuda.current_stream().cuda_stream, w.B, w.C, w.S, w.E,
                                  host_addr, stride, st["dev"].data_ptr(), st["pt"].data_ptr(),
                                  st["tok"].data_ptr(), st["lu"].data_ptr(), st["step"].data_ptr(),
                                  sel.data_ptr(), sel.shape[1], out.data_ptr(), miss.data_ptr(),
                                  status.data_ptr())


def test_noalloc_matches_resolve_call_after_call():
    hs.build()
    tracegen.build()
    lib = hs.load_library()
    w = tracegen.WORKLOADS["dsa"]  # 32 requests x 4096 slots: 1 MiB of the 2 MiB scratch
    T = 6
    ref = hs.Context(w.B, w.C, w.S, w.E)
    tracegen.fill_kv(ref.host_kv_address(), ref.host_stride, w)
    # the caller-owned state of an empty cache
    st = {
        "pt": torch.full((w.B, w.C), -1, dtype=torch.int32, device="cuda"),
        "tok": torch.full((w.B, w.S), -1, dtype=torch.int32, device="cuda"),
        "lu": torch.full((w.B, w.S), -1, dtype=torch.int32, device="cuda"),
        "step": torch.zeros(w.B, dtype=torch.int32, device="cuda"),
        "dev": torch.zeros((w.B, w.S, w.E), dtype=torch.uint8, device="cuda"),
    }
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = torch.from_numpy(tracegen.trace(w, T=T)).cuda()
    out_a = torch.empty_like(sel)
    out_b = torch.empty_like(sel)
    miss_a = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
    miss_b = torch.empty((T, w.B), dtype=torch.int32, device="cuda")
    for t in range(T):
        ref.resolve(sel[t], out_a[t], miss_a[t])
        # under unified addressing the pinned host store's host pointer is device-visible
        rc = _noalloc(lib, w, ref.host_kv_address(), ref.host_stride, st, sel[t], out_b[t],
                      miss_b[t], status)
        assert rc == hs.HS_OK, hs.last_error()
        torch.cuda.synchronize()
        assert torch.equal(out_a[t], out_b[t]), t
        assert torch.equal(miss_a[t], miss_b[t]), t
        assert torch.equal(ref.page_table(), st["pt"]), t
        assert torch.equal(ref.slot_token(), st["tok"]), t
        assert torch.equal(ref.last_use(), st["lu"]), t
        assert torch.equal(ref.step(), st["step"]), t
        assert torch.equal(ref.device_kv(), st["dev"]), t
    assert int(miss_b[1:].sum()) > 0  # later calls had misses to fetch, not only the first
    assert int(status.item()) == 0

    # sizes beyond the fixed scratch array are refused before anything is enqueued
    big = tracegen.Workload("big", 9, B=64, L=1, C=w.C, S=w.S, k=w.k, E=w.E,
                            kv_kind=tracegen.KV_RAW, T=1, keep_pct=90, zipf_s=1.1)
    rc = lib.hs_resolve_noalloc(None, big.B, big.C, big.S, big.E, ref.host_kv_address(),
                                ref.host_stride, st["dev"].data_ptr(), st["pt"].data_ptr(),
                                st["tok"].data_ptr(), st["lu"].data_ptr(), st["step"].data_ptr(),
                                sel[0].data_ptr(), w.k, out_b[0].data_ptr(), miss_b[0].data_ptr(),
                                None)
    assert rc == hs.HS_ERR_LIMIT
    assert "scratch" in hs.last_error()
    torch.cuda.synchronize()
    assert torch.equal(ref.step(), st["step"])
    ref.close()


def test_noalloc_callers_with_separate_state_can_alternate():
    """Two callers (say two layers) each own their state and take turns; the library's
    shared scratch must not leak one caller's hand-off into the other's call."""
    hs.build()
    tracegen.build()
    lib = hs.load_library()
    w = tracegen.WORKLOADS["dsa"]
    B, T = 4, 6
    refs = [hs.Context(B, w.C, w.S, w.E) for _ in range(2)]
    for layer, ref in enumerate(refs):
        tracegen.fill_kv(ref.host_kv_address(), ref.host_stride, w, B=B, layer=layer)
    states = [{
        "pt": torch.full((B, w.C), -1, dtype=torch.int32, device="cuda"),
        "tok": torch.full((B, w.S), -1, dtype=torch.int32, device="cuda"),
        "lu": torch.full((B, w.S), -1, dtype=torch.int32, device="cuda"),
        "step": torch.zeros(B, dtype=torch.int32, device="cuda"),
        "dev": torch.zeros((B, w.S, w.E), dtype=torch.uint8, device="cuda"),
    } for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = torch.from_numpy(tracegen.trace(w, T=T, B=B)).cuda()
    wb = tracegen.Workload("dsa4", w.config, B=B, L=1, C=w.C, S=w.S, k=w.k, E=w.E, kv_kind=w.kv_kind,
                           T=T, keep_pct=w.keep_pct, zipf_s=w.zipf_s)
    for t in range(T):
        for layer in range(2):  # same step count, same selection: tags coincide on purpose
            a_out, b_out = torch.empty_like(sel[t]), torch.empty_like(sel[t])
            a_miss = torch.empty(B, dtype=torch.int32, device="cuda")
            b_miss = torch.empty(B, dtype=torch.int32, device="cuda")
            refs[layer].resolve(sel[t], a_out, a_miss)
            rc = _noalloc(lib, wb, refs[layer].host_kv_address(), refs[layer].host_stride, states[layer],
                          sel[t], b_out, b_miss, status)
            assert rc == hs.HS_OK, hs.last_error()
            torch.cuda.synchronize()
            assert torch.equal(a_out, b_out) and torch.equal(a_miss, b_miss), (t, layer)
            assert torch.equal(refs[layer].device_kv(), states[layer]["dev"]), (t, layer)
    assert int(status.item()) == 0
    for ref in refs:
        ref.close()


def test_noalloc_callers_of_different_sizes_can_alternate():
    """Callers of different sizes share the library's scratch array, whose layout (the miss
    lists, the per-request flags and the fetch counters) then shifts from one call to the
    next. Two such callers -- 4 requests of 4096 slots and 24 requests of 2048 slots --
    take turns, and every output, table and device byte must match hs_resolve on
    contexts of the same sizes."""
    hs.build()
    tracegen.build()
    lib = hs.load_library()
    base = tracegen.WORKLOADS["dsa"]
    T = 6
    shapes = [dict(B=4, S=4096), dict(B=24, S=2048)]
    callers = []
    for i, sh in enumerate(shapes):
        w = tracegen.Workload(f"size{i}", 20 + i, B=sh["B"], L=1, C=base.C, S=sh["S"], k=base.k, E=base.E,
                              kv_kind=base.kv_kind, T=T, keep_pct=base.keep_pct, zipf_s=base.zipf_s,
                              recent=base.recent, seed=40 + i)
        ref = hs.Context(w.B, w.C, w.S, w.E)
        tracegen.fill_kv(ref.host_kv_address(), ref.host_stride, w)
        st = {
            "pt": torch.full((w.B, w.C), -1, dtype=torch.int32, device="cuda"),
            "tok": torch.full((w.B, w.S), -1, dtype=torch.int32, device="cuda"),
            "lu": torch.full((w.B, w.S), -1, dtype=torch.int32, device="cuda"),
            "step": torch.zeros(w.B, dtype=torch.int32, device="cuda"),
            "dev": torch.zeros((w.B, w.S, w.E), dtype=torch.uint8, device="cuda"),
        }
        sel = torch.from_numpy(tracegen.trace(w, T=T)).cuda()
        callers.append((w, ref, st, sel))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(T):
        for w, ref, st, sel in callers:  # alternate sizes call after call
            a_out, b_out = torch.empty_like(sel[t]), torch.full_like(sel[t], -7)
            a_miss = torch.empty(w.B, dtype=torch.int32, device="cuda")
            b_miss = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
            ref.resolve(sel[t], a_out, a_miss)
            rc = _noalloc(lib, w, ref.host_kv_address(), ref.host_stride, st, sel[t], b_out, b_miss, status)
            assert rc == hs.HS_OK, hs.last_error()
            torch.cuda.synchronize()
            assert torch.equal(a_out, b_out) and torch.equal(a_miss, b_miss), (t, w.name)
            for name, key in (("page_table", "pt"), ("slot_token", "tok"), ("last_use", "lu"), ("step", "step"),
                              ("device_kv", "dev")):
                assert torch.equal(getattr(ref, name)(), st[key]), (t, w.name, name)
    assert int(status.item()) == 0
    for _, ref, _, _ in callers:
        ref.close()
