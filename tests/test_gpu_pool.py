"""Pooled contexts on the GPU: requests of different lengths share one pinned host pool
through extents reserved by the pool's first-fit admission, against the oracle.

Each request's history is its own extent of the pool (the oracle gets that extent as
the request's host rows and the extent's length as the request's length); positions past
a request's length are out of range; a request re-admitted into a row starts empty; a
decode-time append lands in the request's extent.
"""
import numpy as np
import pytest
import torch

import hierarchical_kv_cache_swap_gb300 as hs
from oracle import Oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    hs.build()
    import oracle
    oracle.build()


def _trace(rng, R, lens, Cmax, k, T):
    """Selections mostly inside each request's length, some past it, some padding."""
    sel = np.empty((T, R, k), dtype=np.int32)
    for t in range(T):
        for b in range(R):
            hi = max(1, lens[b])
            row = rng.choice(min(Cmax, hi + hi // 8 + 1), size=k, replace=False).astype(np.int32)
            if t % 5 == 4:
                row[: k // 4] = -1
            sel[t, b] = row
    return sel


def test_pooled_requests_of_different_lengths():
    rng = np.random.default_rng(1)
    R, Cmax, S, E, k, T = 6, 3000, 256, 656, 96, 40
    rows = 30000
    pool_mem = torch.empty(rows * E, dtype=torch.uint8).pin_memory()
    pool_np = pool_mem.numpy().reshape(rows, E)
    pool_np[:] = rng.integers(0, 256, size=pool_np.shape, dtype=np.uint8)
    pool = hs.Pool(rows)
    lens = [int(rng.integers(200, Cmax)) for _ in range(R)]
    bases, spacers = [], []
    for n in lens:  # extents scattered between spacers that are released afterwards
        spacers.append(pool.reserve(int(rng.integers(1, 700))))
        b = pool.reserve(n)
        assert b >= 0
        bases.append(b)
    for sp in spacers:
        pool.release(sp)
    assert pool.free_rows() == rows - sum(lens)
    ctx = hs.Context(R, Cmax, S, E, pool=(pool_mem.data_ptr(), rows, E))
    ctx.set_extents(bases, lens)
    orc = Oracle(R, Cmax, S, E)
    for b in range(R):
        orc.set_len(b, int(lens[b]))
    addr = pool_mem.data_ptr()

    def step(sel_t):
        sd = torch.from_numpy(sel_t).cuda()
        out = torch.empty_like(sd)
        miss = torch.empty(R, dtype=torch.int32, device="cuda")
        ctx.resolve(sd, out, miss)
        st = 0
        for b in range(R):
            o_out, o_m, rc = orc.resolve_request(b, addr + bases[b] * E, E, sel_t[b])
            st |= rc
            assert np.array_equal(out[b].cpu().numpy(), o_out), b
            assert int(miss[b]) == o_m, b
        return st

    sel = _trace(rng, R, lens, Cmax, k, T)
    statuses = 0
    for t in range(T // 2):
        statuses |= step(sel[t])
    torch.cuda.synchronize()
    assert statuses & 1 and ctx.status() & hs.HS_STATUS_RANGE  # positions past a length
    # request 2 finishes; a new, longer request is admitted into its row
    pool.release(bases[2])
    lens[2] = 2900
    bases[2] = pool.reserve(2900)
    assert bases[2] >= 0
    ctx.set_extents(bases, lens)
    orc.reset_request(2)
    orc.set_len(2, 2900)
    sel2 = _trace(rng, R, lens, Cmax, k, T)
    for t in range(T // 2, T):
        step(sel2[t])
    # decode-time append into the extents
    torch.cuda.synchronize()
    pool_before = np.ascontiguousarray(pool_np.copy())
    pos = np.array([min(int(lens[b]) - 1, 100 + b) for b in range(R)], dtype=np.int32)
    new = rng.integers(0, 256, size=(R, E), dtype=np.uint8)
    ctx.append(torch.from_numpy(new).cuda(), torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    ref_pool = pool_before  # the oracle appends into its own copy of the pool
    for b in range(R):
        assert orc.append_request(b, ref_pool[bases[b]:], E, int(pos[b]), new[b]) == 0
    assert np.array_equal(pool_np, ref_pool)
    assert np.array_equal(ctx.device_kv().cpu().numpy(), orc.dev)
    for name, ref in (("page_table", orc.pt), ("slot_token", orc.tok), ("last_use", orc.lu), ("step", orc.t)):
        assert np.array_equal(getattr(ctx, name)().cpu().numpy(), ref), name
    ctx.close()
    pool.close()


def test_pooled_context_rejects_bad_extents():
    rows, E = 100, 656
    pool_mem = torch.empty(rows * E, dtype=torch.uint8).pin_memory()
    ctx = hs.Context(2, 50, 16, E, pool=(pool_mem.data_ptr(), rows, E))
    for base, length in (([0, 90], [10, 20]), ([-1, 0], [1, 1]), ([0, 0], [51, 1])):
        with pytest.raises(hs.HsError):
            ctx.set_extents(base, length)
    ctx.set_extents([0, 50], [50, 50])
    ctx.close()
    plain = hs.Context(1, 8, 4, 16)
    with pytest.raises(hs.HsError):
        plain.set_extents([0], [1])
    plain.close()


def test_pooled_resolution_in_a_cuda_graph():
    """A pooled context's resolutions captured in a graph and replayed equal the eager ones
    of a second pooled context over the same pool and extents."""
    rng = np.random.default_rng(4)
    R, Cmax, S, E, k, T = 3, 800, 128, 656, 64, 8
    rows = 4000
    pool_mem = torch.empty(rows * E, dtype=torch.uint8).pin_memory()
    pool_mem.numpy()[:] = rng.integers(0, 256, size=rows * E, dtype=np.uint8)
    lens = [700, 300, 800]
    bases = [2500, 40, 1200]
    sel = torch.from_numpy(_trace(rng, R, lens, Cmax, k, T)).cuda()
    outs = []
    for graph in (False, True):
        ctx = hs.Context(R, Cmax, S, E, pool=(pool_mem.data_ptr(), rows, E))
        ctx.set_extents(bases, lens)
        out = torch.full((T, R, k), -9, dtype=torch.int32, device="cuda")
        miss = torch.empty((T, R), dtype=torch.int32, device="cuda")
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for t in range(T):
                        ctx.resolve(sel[t], out[t], miss[t], stream=s)
            torch.cuda.current_stream().wait_stream(s)
            g.replay()
        else:
            for t in range(T):
                ctx.resolve(sel[t], out[t], miss[t])
        torch.cuda.synchronize()
        outs.append((out.clone(), miss.clone(), ctx.page_table().clone(), ctx.device_kv().clone()))
        ctx.close()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
