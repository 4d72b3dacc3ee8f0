"""The shared host pool, the capacity planner, and the oracle's per-request lengths.

Host logic only (no GPU): the library's pool bookkeeping against an independently
written first-fit interval model; the planner against the oracle's plain restatement,
against a deployment example of the pages worked by hand, and against invariants; the
oracle's per-request length against a context of that many positions.
"""
import random

import numpy as np
import pytest

import hierarchical_kv_cache_swap_gb300 as hs
from oracle.plan import plan as plan_ref


class IntervalModel:
    """First fit over a sorted list of free (base, length) intervals."""

    def __init__(self, rows):
        self.free = [(0, rows)]
        self.used = {}

    def reserve(self, n):
        for i, (b, l) in enumerate(self.free):
            if l >= n:
                self.free[i:i + 1] = [(b + n, l - n)] if l > n else []
                self.used[b] = n
                return b
        return -1

    def release(self, b):
        n = self.used.pop(b)
        self.free.append((b, n))
        self.free.sort()
        merged = []
        for fb, fl in self.free:
            if merged and merged[-1][0] + merged[-1][1] == fb:
                merged[-1] = (merged[-1][0], merged[-1][1] + fl)
            else:
                merged.append((fb, fl))
        self.free = merged

    def free_rows(self):
        return sum(l for _, l in self.free)

    def largest(self):
        return max((l for _, l in self.free), default=0)


def test_pool_matches_first_fit_model():
    hs.build()
    for seed in range(4):
        rng = random.Random(seed)
        rows = rng.choice([100, 1000, 65536])
        pool, model = hs.Pool(rows), IntervalModel(rows)
        live = []
        for _ in range(400):
            if live and rng.random() < 0.45:
                b = live.pop(rng.randrange(len(live)))
                pool.release(b)
                model.release(b)
            else:
                n = rng.randint(1, max(1, rows // 6))
                got, want = pool.reserve(n), model.reserve(n)
                assert got == want, (seed, n)
                if got >= 0:
                    live.append(got)
            assert pool.free_rows() == model.free_rows()
            assert pool.largest_free() == model.largest()
        for b in live:
            pool.release(b)
        assert pool.free_rows() == rows and pool.largest_free() == rows  # fully merged again
        with pytest.raises(hs.HsError):
            pool.release(rows + 5)
        assert pool.reserve(rows + 1) == -1 and pool.reserve(0) == -1
        pool.close()


EXAMPLE = dict(top_k=2048, device_buffer_size=6144, host_to_device_ratio=10.0, entry_bytes=656, layers=61,
               context_len=40960, hbm_bytes=100 * 2 ** 30, host_bytes=1500 * 2 ** 30, miss_fraction=0.06,
               link_gbs=200.0)


def test_plan_deployment_example_by_hand():
    """The disaggregated-decode knobs (top_k 2048, buffer 6144, ratio 10), a 61-layer model
    with 656-byte entries, 32k + 8k contexts, 100 GiB of HBM and 1500 GiB of pinned host
    memory. By hand: per layer 6144*656 + 4*40960 + 28*6144 + 268 = 4,030,464 + 163,840 +
    172,032 + 268 = 4,366,604 B, so 266,362,844 B per request and floor(107,374,182,400 /
    266,362,844) = 403 requests by HBM; the pool wants 10*403*6144 = 24,760,320 rows and
    1500 GiB holds floor(1,610,612,736,000 / (61*656)) = 40,249,218 rows, so 24,760,320
    rows = floor(604.5) = 604 histories of 40960 positions; 403 requests are admitted.
    (The per-layer device bytes are what hs_create allocates: measured on a GPU in
    tests/test_gpu_plan.py.)"""
    r = hs.plan(**EXAMPLE)
    assert r["device_bytes_per_request"] == 266_362_844
    assert r["requests_by_device"] == 403
    assert r["host_pool_rows"] == 24_760_320
    assert r["requests_by_host"] == 604
    assert r["requests"] == 403
    assert r["miss_bytes_per_step"] == pytest.approx(403 * 61 * 0.06 * 2048 * 656)
    assert r["link_us_per_step"] == pytest.approx(r["miss_bytes_per_step"] / 200e3)


def test_plan_matches_restatement_and_invariants():
    rng = random.Random(3)
    for _ in range(300):
        k = rng.choice([128, 512, 2048, 4096])
        p = dict(top_k=k, device_buffer_size=k * rng.choice([1, 2, 3, 4]),
                 host_to_device_ratio=rng.choice([1.0, 2.5, 8.0, 10.0]), entry_bytes=rng.choice([656, 1152, 65536]),
                 layers=rng.randint(1, 80), context_len=rng.randint(k, 1 << 20),
                 hbm_bytes=rng.randint(0, 250 << 30), host_bytes=rng.randint(0, 2 << 40),
                 miss_fraction=rng.random(), link_gbs=rng.choice([0.0, 64.0, 200.0]))
        r = hs.plan(**p)
        # the device footprint is pinned by measurement on a GPU; here it is an input
        ref = plan_ref(**p, device_bytes_per_layer=r["device_bytes_per_request"] // p["layers"])
        for key, v in ref.items():
            assert r[key] == pytest.approx(v, rel=1e-12, abs=1e-9), key
        assert r["requests"] == min(r["requests_by_device"], r["requests_by_host"])
        assert r["host_pool_rows"] <= p["host_to_device_ratio"] * r["requests_by_device"] * p["device_buffer_size"]
        more = hs.plan(**{**p, "hbm_bytes": p["hbm_bytes"] * 2})
        assert more["requests_by_device"] >= r["requests_by_device"]
    for bad in ({"device_buffer_size": 1024}, {"host_to_device_ratio": 0.0}, {"miss_fraction": 1.5}):
        with pytest.raises(hs.HsError):
            hs.plan(**{**EXAMPLE, **bad})


def run_length_limit(Oracle, lib_path=None):
    """A request limited to n positions resolves exactly like a context of n positions
    (positions >= n are out of range in both); a reset request behaves like a new one."""
    rng = np.random.default_rng(9)
    n, Cbig, S, E, k = 40, 100, 12, 16, 6
    host = rng.integers(0, 256, size=(1, Cbig, E), dtype=np.uint8)
    big = Oracle(1, Cbig, S, E, lib_path=lib_path)
    big.set_len(0, n)
    small = Oracle(1, n, S, E, lib_path=lib_path)
    for t in range(30):
        sel = rng.choice(60, size=(1, k), replace=False).astype(np.int32)  # some >= n
        o1, m1, st1 = big.resolve(host, E, sel)
        o2, m2, st2 = small.resolve(host[:, :n].copy(), E, sel)
        assert np.array_equal(o1, o2) and np.array_equal(m1, m2) and st1 == st2, t
        assert np.array_equal(big.tok, small.tok) and np.array_equal(big.lu, small.lu)
        assert np.array_equal(big.pt[:, :n], small.pt) and (big.pt[:, n:] == -1).all()
        assert np.array_equal(big.dev, small.dev)
    big.reset_request(0)
    fresh = Oracle(1, Cbig, S, E, lib_path=lib_path)
    fresh.set_len(0, n)
    sel = rng.choice(n, size=(1, k), replace=False).astype(np.int32)
    a, b = big.resolve(host, E, sel), fresh.resolve(host, E, sel)
    assert np.array_equal(a[0], b[0]) and np.array_equal(big.dev, fresh.dev) and np.array_equal(big.t, fresh.t)


def test_oracle_length_limit(oracle_mod):
    run_length_limit(oracle_mod.Oracle)
