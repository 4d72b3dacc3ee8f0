"""Bit-exact parity of the CUDA path (through the C ABI) with the CPU oracle.

The oracle's rule is the deterministic LRU reading of the HiSparse paper abstract
(hit detection, LRU replacement, host-to-device fetch per layer) and of the blog
commentary's sections two and three (hits used in place, misses swapped in over an
LRU victim, the page table updated in the same step). Everything compared is
integer or byte data, so the bar is exact equality.
"""
import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
import tracegen
from oracle import Oracle
from tests.gpu_harness import DeviceRun, run_and_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    hs.build()
    tracegen.build()
    import oracle
    oracle.build()
    torch.cuda.init()


# ------------------------------------------------------------------ the five workloads

def test_tiny_full_trace():
    w = tracegen.WORKLOADS["tiny"]
    run_and_compare(w, T=w.T, checkpoints=range(0, w.T, 4))


def test_dsa_full_trace_all_requests():
    w = tracegen.WORKLOADS["dsa"]
    run_and_compare(w, T=w.T, checkpoints=[0, 1, 17, 64, 128, w.T - 1])


@pytest.mark.parametrize("S", [2048, 4096, 6144])
@pytest.mark.parametrize("keep", [50, 80, 95])
def test_sweep_point_sampled(S, keep):
    w = tracegen.sweep_workload(S, keep)
    sample = [0, 1, 13, 31, 32, 50, 62, 63]
    run_and_compare(w, T=w.T, sample=sample, checkpoints=[0, 5, w.T - 1])


def test_long_context_full_size_sampled():
    """256 requests x 131072 positions (22 GB of pinned host KV), sampled requests."""
    w = tracegen.WORKLOADS["long"]
    sample = [0, 1, 77, 128, 200, 254, 255]
    run_and_compare(w, T=w.T, sample=sample, checkpoints=[0, 1, 31, w.T - 1])


def test_quest_pages_eight_layers_full_size():
    """Quest-style 64-KiB pages at full size: 64 requests x 4096 pages (17.2 GB of pinned
    host KV per layer), 256-page buffers, k = 128, the whole 128-step trace, every request
    compared. The 8 layers share every selection and are independent contexts, so they are
    resolved one after the other, each over its own store, freed before the next."""
    w = tracegen.WORKLOADS["quest"]
    B, T = w.B, w.T
    sel = tracegen.trace(w, T=T, B=B)
    for layer in range(w.L):
        run = DeviceRun(w, T, B=B, layer=layer, sel=sel)
        stats = run_and_compare(w, T=T, B=B, checkpoints=[0, 7, T - 1], layer=layer, run=run)
        assert stats["misses"].sum() > 0
        run.close()


# ------------------------------------------------------------------ replacement policies

@pytest.mark.parametrize("policy", [hs.POLICY_FIFO, hs.POLICY_RANDOM])
def test_policy_dsa_full_trace_all_requests(policy):
    w = tracegen.WORKLOADS["dsa"]
    run_and_compare(w, T=64, checkpoints=[0, 1, 17, 63], policy=policy, seed=0x5EED)


@pytest.mark.parametrize("policy", [hs.POLICY_FIFO, hs.POLICY_RANDOM])
@pytest.mark.parametrize("C,S,k,E,B", [(37, 5, 5, 16, 3), (300, 33, 7, 48, 2), (100000, 777, 513, 144, 5)])
def test_policy_ragged_shapes(policy, C, S, k, E, B):
    w = tracegen.Workload("ragged", 9, B=B, L=1, C=C, S=S, k=k, E=E, kv_kind=tracegen.KV_RAW,
                          T=40, keep_pct=60, zipf_s=1.1, seed=C)
    run_and_compare(w, T=w.T, checkpoints=[0, 1, 19, 39], policy=policy, seed=C * 7919)


def test_policy_random_sampled_requests_use_their_own_draws():
    """Sampled requests (oracle rows standing for request numbers 3, 40, 63) draw the
    keys of their own request numbers."""
    w = tracegen.sweep_workload(4096, 80)
    run_and_compare(w, T=24, sample=[3, 40, 63], checkpoints=[0, 23], policy=hs.POLICY_RANDOM, seed=1)


def test_policy_switch_mid_trace():
    """The state carries over when the policy changes between calls."""
    w = tracegen.WORKLOADS["tiny"]
    T = 30
    run = DeviceRun(w, T)
    o = Oracle(run.B, w.C, w.S, w.E)
    host = run.ctx.host_kv()
    for t in range(T):
        policy = (hs.POLICY_LRU, hs.POLICY_FIFO, hs.POLICY_RANDOM)[(t // 7) % 3]
        run.ctx.set_policy(policy, 77)
        o.set_policy(policy, 77)
        run.step(t)
        o_out, o_miss, _ = o.resolve(host, run.ctx.host_stride, run.sel[t])
        assert np.array_equal(run.out_dev[t].cpu().numpy(), o_out), t
        assert np.array_equal(run.miss_dev[t].cpu().numpy(), o_miss), t
    torch.cuda.synchronize()
    for name, ref in (("page_table", o.pt), ("slot_token", o.tok), ("last_use", o.lu), ("step", o.t)):
        assert np.array_equal(getattr(run.ctx, name)().cpu().numpy(), ref), name
    assert np.array_equal(run.ctx.device_kv().cpu().numpy(), o.dev)
    with pytest.raises(RuntimeError):
        run.ctx.set_policy(3)
    run.close()


# ------------------------------------------------------------------ properties and edge cases

def test_noio_all_hits_after_first_call():
    w = tracegen.noio_workload(4096)
    run = DeviceRun(w, T=12, fill=False)
    for t in range(12):
        run.step(t)
    miss = run.miss_dev.cpu().numpy()
    assert (miss[0] == w.k).all() and (miss[1:] == 0).all()
    run.close()


def test_calls_alternating_all_hit_and_missing_with_padding():
    """Every selection row is resolved twice in a row, the second time in a new order with
    some entries turned into padding: the repeat is all hits (or padding), and the next
    call has hits, misses and padding after an all-hit call. Hits and padding are answered
    either by the probe itself or after the hand-off flags, depending on the previous
    call; both orders must give the oracle's results, tables and bytes."""
    w = tracegen.WORKLOADS["dsa"]
    B, T = 6, 12
    base = tracegen.trace(w, T=T // 2, B=B)
    rng = np.random.default_rng(17)
    rows = []
    for t in range(T // 2):
        rows.append(base[t].copy())
        rep = np.stack([rng.permutation(r) for r in base[t]])
        rep[:, :rng.integers(0, 40)] = -1  # a few padding entries
        rows.append(rep.astype(np.int32))
    sel = np.stack(rows)
    run = DeviceRun(w, T, B=B, sel=sel)
    stats = run_and_compare(w, T=T, B=B, run=run, checkpoints=[0, 1, 5, T - 1])
    miss = run.miss_dev.cpu().numpy()
    assert (miss[1::2] == 0).all() and (miss[2::2] > 0).all()
    assert stats["misses"].sum() > 0
    run.close()


@pytest.mark.parametrize("C,S,k,E,B", [
    (1, 1, 1, 16, 1),          # degenerate: one position, one slot
    (37, 5, 5, 16, 3),         # k = S, ragged bitmap words
    (300, 33, 7, 48, 2),       # S not a multiple of 32
    (2049, 2047, 2047, 32, 2), # k = S just below a power of two, C ragged past a group
    (100000, 777, 513, 144, 5),
    (20000, 6000, 5000, 32, 2),  # k above one probe batch of 4 x 512: batched probe and re-read answers
])
def test_random_shapes_and_ragged_tails(C, S, k, E, B):
    w = tracegen.Workload("ragged", 9, B=B, L=1, C=C, S=S, k=k, E=E, kv_kind=tracegen.KV_RAW,
                          T=40, keep_pct=60, zipf_s=1.1, seed=C)
    run_and_compare(w, T=w.T, checkpoints=[0, 1, 19, 39])


def _custom_run(C, S, E, rows):
    """rows: list of [B][k] selections (same k); returns (gpu outs, gpu misses, ctx, oracle)."""
    B, k = len(rows[0]), len(rows[0][0])
    ctx = hs.Context(B, C, S, E)
    host = ctx.host_kv()
    host[:] = np.random.default_rng(C).integers(0, 256, size=host.shape, dtype=np.uint8)
    o = Oracle(B, C, S, E)
    for t, r in enumerate(rows):
        sel = np.asarray(r, dtype=np.int32)
        sd = torch.from_numpy(sel).cuda()
        out = torch.empty_like(sd)
        miss = torch.empty(B, dtype=torch.int32, device="cuda")
        ctx.resolve(sd, out, miss)
        o_out, o_miss, _ = o.resolve(host, ctx.host_stride, sel)
        assert np.array_equal(out.cpu().numpy(), o_out), t
        assert np.array_equal(miss.cpu().numpy(), o_miss), t
    torch.cuda.synchronize()
    for name, ref in (("page_table", o.pt), ("slot_token", o.tok), ("last_use", o.lu), ("step", o.t)):
        assert np.array_equal(getattr(ctx, name)().cpu().numpy(), ref), name
    assert np.array_equal(ctx.device_kv().cpu().numpy(), o.dev)
    return ctx, o


def test_wide_stamp_range_needs_several_radix_passes():
    """Candidates whose stamps span > 2^8 and > 2^16 calls (2 and 3 LSD digit passes)."""
    C, S, E = 64, 10, 16
    rows = [[[p, 40 + p]] for p in range(10)]      # fill: two positions per call, k = 2
    rows += [[[0, 40]]] * 300                        # 300 all-hit calls on slots 0/1
    rows += [[[1, 50]], [[2, 51]], [[60, 61]]]       # misses over stamps spread by ~300
    ctx, _ = _custom_run(C, S, E, rows)
    ctx.close()
    rows = [[[p, 40 + p]] for p in range(10)] + [[[0, 40]]] * 70000 + [[[1, 50]], [[62, 63]]]
    ctx, _ = _custom_run(C, S, E, rows)
    ctx.close()


def test_padding_out_of_range_and_duplicates_set_status():
    C, S, E = 50, 8, 16
    rows = [[[3, -1, 3, 99], [5, 6, 7, 8]], [[-5, 3, 4, -1], [9, 8, 8, -3]]]
    ctx = hs.Context(2, C, S, E)
    host = ctx.host_kv()
    host[:] = 7
    o = Oracle(2, C, S, E)
    status = 0
    for r in rows:
        sel = np.asarray(r, dtype=np.int32)
        sd = torch.from_numpy(sel).cuda()
        out = torch.empty_like(sd)
        miss = torch.empty(2, dtype=torch.int32, device="cuda")
        ctx.resolve(sd, out, miss)
        o_out, o_miss, st = o.resolve(host, E, sel)
        status |= st
        assert np.array_equal(out.cpu().numpy(), o_out)
        assert np.array_equal(miss.cpu().numpy(), o_miss)
    assert ctx.status() == status == hs.HS_STATUS_RANGE | hs.HS_STATUS_DUP
    ctx.clear_status()
    assert ctx.status() == 0
    ctx.close()


def test_permutation_invariance():
    w = tracegen.WORKLOADS["tiny"]
    a = DeviceRun(w, T=20)
    b = DeviceRun(w, T=20)
    rng = np.random.default_rng(1)
    perms = [rng.permutation(w.k) for _ in range(20)]
    b.sel_dev = torch.from_numpy(np.stack([a.sel[t][:, perms[t]] for t in range(20)])).cuda()
    for t in range(20):
        a.step(t)
        b.step(t)
    oa, ob = a.out_dev.cpu().numpy(), b.out_dev.cpu().numpy()
    for t in range(20):
        assert np.array_equal(oa[t][:, perms[t]], ob[t])
    for name in ("page_table", "slot_token", "last_use", "step", "device_kv"):
        assert torch.equal(getattr(a.ctx, name)(), getattr(b.ctx, name)())
    a.close()
    b.close()


def test_graph_replay_equals_eager():
    """The step can be captured in a CUDA graph; replays advance the state like eager calls."""
    w = tracegen.WORKLOADS["dsa"]
    T = 24
    eager = DeviceRun(w, T, B=8)
    graph = DeviceRun(w, T, B=8)
    for t in range(T):
        eager.step(t)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for t in range(T // 2):
                graph.step(t, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    # capture enqueued nothing; replay twice over the two halves of the trace
    g.replay()
    torch.cuda.synchronize()
    first = graph.out_dev[: T // 2].clone()
    graph.sel_dev[: T // 2].copy_(graph.sel_dev[T // 2:].clone())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(first, eager.out_dev[: T // 2])
    assert torch.equal(graph.out_dev[: T // 2], eager.out_dev[T // 2:])
    assert torch.equal(graph.miss_dev[: T // 2], eager.miss_dev[T // 2:])
    for name in ("page_table", "slot_token", "last_use", "step", "device_kv"):
        assert torch.equal(getattr(eager.ctx, name)(), getattr(graph.ctx, name)()), name
    eager.close()
    graph.close()


def _host_buffer(shape, pinned):
    if pinned:  # page-locked: the kernels read or write it in place
        return torch.empty(shape, dtype=torch.int32).pin_memory().numpy()
    return np.empty(shape, dtype=np.int32)  # pageable: staged through device buffers


@pytest.mark.parametrize("sel_pinned,out_pinned", [(False, False), (True, True), (True, False), (False, True)])
def test_host_buffer_entry_point_matches_device_entry_point(sel_pinned, out_pinned):
    w = tracegen.WORKLOADS["dsa"]
    T = 10
    a = DeviceRun(w, T, B=4)
    b = hs.Context(4, w.C, w.S, w.E)
    tracegen.fill_kv(b.host_kv_address(), b.host_stride, w, B=4)
    sel = _host_buffer(a.sel.shape, sel_pinned)
    sel[...] = a.sel
    out = _host_buffer((4, w.k), out_pinned)
    miss = _host_buffer((4,), out_pinned)
    out[...] = -7
    for t in range(T):
        a.step(t)
        b.resolve_host(sel[t], out, miss)
        torch.cuda.synchronize()
        assert np.array_equal(out, a.out_dev[t].cpu().numpy())
        assert np.array_equal(miss, a.miss_dev[t].cpu().numpy())
    assert torch.equal(a.ctx.device_kv(), b.device_kv())
    a.close()
    b.close()


@pytest.mark.parametrize("B", [32, 200])
def test_serialised_kernels_equal_the_overlapped_ones(B):
    """hs_resolve overlaps its two kernels when there are at most as many requests as SMs
    (the fetch waits for each request's flags) and runs them one after the other beyond;
    the per-kernel timing entry point always runs them one after the other, with events
    between. Every way must give the oracle's results."""
    w = tracegen.Workload("split", 14, B=B, L=1, C=4096, S=512, k=256, E=64, kv_kind=tracegen.KV_RAW,
                          T=12, keep_pct=80, zipf_s=1.1, seed=B)
    a = DeviceRun(w, T=w.T)
    run_and_compare(w, T=w.T, run=a, checkpoints=[0, w.T - 1])
    b = DeviceRun(w, T=w.T)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for t in range(w.T):
        b.ctx.resolve_profiled(b.sel_dev[t], b.out_dev[t], b.miss_dev[t], ev)
    torch.cuda.synchronize()
    assert b.ctx.status() == 0
    assert torch.equal(a.out_dev, b.out_dev) and torch.equal(a.miss_dev, b.miss_dev)
    for name in ("page_table", "slot_token", "last_use", "step", "device_kv"):
        assert torch.equal(getattr(a.ctx, name)(), getattr(b.ctx, name)()), name
    a.close()
    b.close()


def test_no_copy_flag_keeps_bookkeeping_and_skips_fetch():
    w = tracegen.WORKLOADS["tiny"]
    a = DeviceRun(w, T=16)
    b = DeviceRun(w, T=16)
    b.ctx.set_flags(hs.HS_FLAG_NO_COPY)
    assert a.ctx.kernels_per_call() == 2 and b.ctx.kernels_per_call() == 1
    for t in range(16):
        a.step(t)
        b.step(t)
    assert torch.equal(a.out_dev, b.out_dev) and torch.equal(a.miss_dev, b.miss_dev)
    for name in ("page_table", "slot_token", "last_use", "step"):
        assert torch.equal(getattr(a.ctx, name)(), getattr(b.ctx, name)())
    assert int(b.ctx.device_kv().count_nonzero()) == 0
    a.close()
    b.close()


def test_reset_restores_empty_state():
    w = tracegen.WORKLOADS["tiny"]
    run = DeviceRun(w, T=8)
    for t in range(8):
        run.step(t)
    run.ctx.reset()
    torch.cuda.synchronize()
    assert (run.ctx.page_table() == -1).all() and (run.ctx.slot_token() == -1).all()
    assert (run.ctx.last_use() == -1).all() and (run.ctx.step() == 0).all()
    assert int(run.ctx.device_kv().count_nonzero()) == 0
    run.close()


def test_bad_calls_enqueue_nothing():
    ctx = hs.Context(2, 100, 10, 16)
    sel = torch.zeros((2, 11), dtype=torch.int32, device="cuda")
    out = torch.empty_like(sel)
    miss = torch.empty(2, dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError, match="k=11"):
        ctx.resolve(sel, out, miss)
    with pytest.raises(hs.HsError, match="B=1"):
        ctx.resolve(sel[:1, :5], out[:1, :5], miss[:1])
    torch.cuda.synchronize()
    assert (ctx.step() == 0).all()
    ctx.close()


def test_contexts_of_different_sizes_coexist():
    """A small context created after a large one must not break the large one's launches."""
    big = tracegen.WORKLOADS["dsa"]
    small = tracegen.Workload("small", 9, B=2, L=1, C=64, S=16, k=8, E=16, kv_kind=tracegen.KV_RAW,
                              T=6, keep_pct=50, zipf_s=1.1, seed=3)
    a = DeviceRun(big, T=6, B=2)
    b = DeviceRun(small, T=6)
    for t in range(6):
        a.step(t)
        b.step(t)
    torch.cuda.synchronize()
    a.close()
    b.close()
    run_and_compare(big, T=6, B=2)
    run_and_compare(small, T=6)


def test_no_copy_calls_interleaved_with_fetching_calls():
    """A call without the fetch (HS_FLAG_NO_COPY) between fetching calls leaves a hand-off
    the next fetch must not mistake for its own: tables, outputs and the rows fetched by
    fetching calls must still match the oracle."""
    w = tracegen.WORKLOADS["dsa"]
    B, T = 4, 24
    run = DeviceRun(w, T, B=B)
    o = Oracle(B, w.C, w.S, w.E)
    base = run.ctx.host_kv_address()
    row_bytes = w.C * run.ctx.host_stride
    fetched = [set() for _ in range(B)]  # slots (re)filled by a fetching call
    for t in range(T):
        no_copy = t % 3 == 1
        run.ctx.set_flags(hs.HS_FLAG_NO_COPY if no_copy else 0)
        run.step(t)
        torch.cuda.synchronize()
        out = run.out_dev[t].cpu().numpy()
        miss = run.miss_dev[t].cpu().numpy()
        tok_before = o.tok.copy()
        for b in range(B):
            o_out, o_m, _ = o.resolve_request(b, base + b * row_bytes, run.ctx.host_stride, run.sel[t, b])
            assert np.array_equal(o_out, out[b]) and o_m == miss[b], (t, b)
            changed = set(np.nonzero(o.tok[b] != tok_before[b])[0].tolist())
            if no_copy:
                fetched[b] -= changed
            else:
                fetched[b] |= changed
    for name, ref in (("page_table", o.pt), ("slot_token", o.tok), ("last_use", o.lu), ("step", o.t)):
        assert np.array_equal(getattr(run.ctx, name)().cpu().numpy(), ref), name
    dev = run.ctx.device_kv().cpu().numpy()
    for b in range(B):
        rows = sorted(fetched[b])
        assert rows, b
        assert np.array_equal(dev[b, rows], o.dev_rows(b)[rows]), b
    assert run.ctx.status() == 0
    run.close()
