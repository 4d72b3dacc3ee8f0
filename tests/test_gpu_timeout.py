"""Every device wait gives up in bounded time, reports it, and leaves the context usable.

The kernels' waits -- the fetch grid waiting for its resolution's per-request flags, the
attention's roles waiting on their shared-memory barriers -- are bounded by the GPU's
global timer: once a CTA has run for the context's wait limit, the wait gives up, sets
HS_STATUS_TIMEOUT and the kernel returns. These tests make a wait run out on purpose
without any fault: HS_FLAG_TEST_STALL makes the resolution publish nothing (so the fetch
waits for flags that are never raised) and the attention's producers withhold their first
fill (so the MMA issuer waits for a barrier that never completes). With a 1 ms limit the
stalled call must take about that long on the GPU -- long enough to show the wait really
waited, short enough to show it gave up -- and after hs_reset the same context must again
agree with the oracle.
"""
import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen
from oracle import Oracle
from tests.gpu_harness import DeviceRun, run_and_compare

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module", autouse=True)
def _built():
    hs.build()
    tracegen.build()
    import oracle
    oracle.build()
    torch.cuda.init()


def gpu_ms(fn) -> float:
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b)


def test_stalled_fetch_wait_times_out_promptly_then_context_recovers():
    w = tracegen.WORKLOADS["dsa"]
    B, T = 4, 8  # 4 requests: the fetch grid overlaps the resolution and waits on its flags
    run = DeviceRun(w, T, B=B)
    ctx = run.ctx
    ctx.set_wait_limit(LIMIT_NS)
    ctx.set_flags(hs.HS_FLAG_TEST_STALL)
    assert ctx.kernels_per_call() == 2
    ms = gpu_ms(lambda: run.step(0))
    assert ctx.status() & hs.HS_STATUS_TIMEOUT
    assert 0.5 <= ms <= 50.0, f"stalled call took {ms:.3f} ms on the GPU with a 1 ms wait limit"
    # the fetch stored nothing: the slots of the cold call are still zero
    assert int(ctx.device_kv().count_nonzero()) == 0
    # a second stalled call runs out the same way (the fetch CTAs' call counters advanced)
    ms2 = gpu_ms(lambda: run.step(1))
    assert 0.5 <= ms2 <= 50.0
    # back to normal: reset, and the whole trace agrees with the oracle bit for bit
    ctx.set_flags(0)
    ctx.set_wait_limit(20_000_000)
    ctx.reset()
    torch.cuda.synchronize()
    assert ctx.status() == 0
    stats = run_and_compare(w, T=T, B=B, run=run, checkpoints=[0, T - 1])
    assert stats["misses"].sum() > 0
    run.close()


def test_wait_limit_is_checked_on_the_host():
    ctx = hs.Context(2, 64, 16, 16)
    for bad in (0, 999, 10_000_000_001):
        with pytest.raises(hs.HsError):
            ctx.set_wait_limit(bad)
    ctx.set_wait_limit(1000)
    ctx.set_wait_limit(10_000_000_000)
    ctx.close()


def test_stalled_attention_times_out_promptly_then_agrees_with_the_oracle():
    w = tracegen.Workload("stall_att", 13, B=2, L=1, C=1024, S=512, k=300, E=656,
                          kv_kind=tracegen.KV_DSA656, T=2, keep_pct=70, zipf_s=1.1, seed=8)
    ctx = hs.Context(w.B, w.C, w.S, w.E)
    tracegen.fill_kv(ctx.host_kv_address(), ctx.host_stride, w)
    sel = tracegen.trace(w, T=w.T)
    o_ref_ctx = Oracle(w.B, w.C, w.S, w.E)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda")
    miss = torch.empty(w.B, dtype=torch.int32, device="cuda")
    for t in range(w.T):
        ctx.resolve(torch.from_numpy(sel[t]).cuda(), out, miss)
        ref_out, _, _ = o_ref_ctx.resolve(ctx.host_kv(), ctx.host_stride, sel[t])
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref_out)
    H, sm = 64, 576 ** -0.5
    q = torch.from_numpy(np.random.default_rng(3).standard_normal((w.B, H, 576)).astype(np.float32))
    q = q.to(torch.bfloat16)
    qd = q.cuda()
    o = torch.empty((w.B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.B, H), dtype=torch.float32, device="cuda")
    nbytes = ctx.attend_workspace(w.B, H, w.k)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None

    ctx.set_wait_limit(LIMIT_NS)
    ctx.set_flags(hs.HS_FLAG_TEST_STALL)
    ms = gpu_ms(lambda: ctx.attend(qd, out, o, lse, sm, workspace=ws))
    assert ctx.status() & hs.HS_STATUS_TIMEOUT
    assert 0.5 <= ms <= 50.0, f"stalled attention took {ms:.3f} ms on the GPU with a 1 ms wait limit"

    ctx.set_flags(0)
    ctx.set_wait_limit(20_000_000)
    ctx.clear_status()
    ctx.attend(qd, out, o, lse, sm, workspace=ws)
    torch.cuda.synchronize()
    assert ctx.status() == 0
    qb = q.view(torch.int16).numpy().view(np.uint16)
    got, got_lse = o.cpu().numpy(), lse.cpu().numpy()
    for b in range(w.B):
        ref, ref_lse, absw = o_ref_ctx.attend(b, qb[b], ref_out[b], sm)
        assert (np.abs(got[b] - ref) <= 2.0 ** -7 * absw + 1e-5).all(), f"attention differs for request {b}"
        assert (np.abs(got_lse[b] - ref_lse) <= 2.0 ** -7 + 1e-5 * np.abs(ref_lse)).all()
    ctx.close()
