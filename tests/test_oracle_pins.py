"""Pins for the CPU oracle: checks against things other than the oracle itself.

Sources of truth (the HiSparse pages fix no worked example, so these are the
properties they do fix, plus textbook results):
  * exactness: every selected entry the consumer reads equals the host row, and
    every selected position is resident after the call (paper abstract: an exact
    cache whose outputs are unchanged because only placement changes);
  * LRU replacement of misses, hits served in place (blog commentary, section two;
    paper abstract) -- checked against a textbook LRU cache (k = 1) and an
    independently written recency-list LRU (any k);
  * a fixed-size per-request cache (paper abstract): never more than S mapped;
  * closed forms: cold start, S >= C (compulsory misses only), S = k, and the
    per-step miss bound k - floor(keep * k) of the locality traces;
  * a trace worked by hand.
"""
import itertools
import random

import numpy as np
import pytest

from tests.lru_models import RecencyListLRU, TextbookFIFO, TextbookLRU, splitmix64

pytestmark = pytest.mark.filterwarnings("ignore")


def _host(R, C, E, seed=0):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(R, C, E), dtype=np.uint8)


# --------------------------------------------------------------------- hand trace

# Worked by hand from the LRU reading (S = 3 slots, C = 8 positions, k = 2):
#   t=0 sel [5,2]: cold; misses ascending 2,5 take slots 0,1 (all stamps -1, slot
#       order) -> out [1,0], tok [2,5,-1], lu [0,0,-1], m 2
#   t=1 sel [7,2]: 2 hits slot 0; non-hit order (-1,s2),(0,s1) -> 7 takes slot 2
#       -> out [2,0], tok [2,5,7], lu [1,0,1], m 1
#   t=2 sel [3,6]: no hit; order (0,s1),(1,s0),(1,s2) -> 3->s1 (evicts 5), 6->s0
#       (evicts 2) -> out [1,0], tok [6,3,7], lu [2,2,1], m 2
#   t=3 sel [7,3]: hits s2, s1 -> out [2,1], lu [2,3,3], m 0
#   t=4 sel [2,0]: no hit; order (2,s0),(3,s1),(3,s2) -> 0->s0 (evicts 6),
#       2->s1 (evicts 3) -> out [1,0], tok [0,2,7], lu [4,4,3], m 2
#   t=5 sel [7,4]: 7 hits s2 (the oldest stamp, but hit slots are not evictable);
#       order of the rest (4,s0),(4,s1) -> 4->s0 (evicts 0) -> out [2,0],
#       tok [4,2,7], lu [5,4,5], m 1
#   t=6 sel [-1,2]: padding + hit s1 -> out [-1,1], lu [5,6,5], m 0
HAND = [
    ([5, 2], [1, 0], [2, 5, -1], [0, 0, -1], 2),
    ([7, 2], [2, 0], [2, 5, 7], [1, 0, 1], 1),
    ([3, 6], [1, 0], [6, 3, 7], [2, 2, 1], 2),
    ([7, 3], [2, 1], [6, 3, 7], [2, 3, 3], 0),
    ([2, 0], [1, 0], [0, 2, 7], [4, 4, 3], 2),
    ([7, 4], [2, 0], [4, 2, 7], [5, 4, 5], 1),
    ([-1, 2], [-1, 1], [4, 2, 7], [5, 6, 5], 0),
]


def run_hand_trace(Oracle, lib_path=None):
    C, S, E = 8, 3, 16
    host = np.arange(C * E, dtype=np.uint32).astype(np.uint8).reshape(1, C, E)
    o = Oracle(1, C, S, E, lib_path=lib_path)
    for t, (sel, out_x, tok_x, lu_x, m_x) in enumerate(HAND):
        out, m, st = o.resolve(host, E, np.array([sel], dtype=np.int32))
        assert out[0].tolist() == out_x, (t, out)
        assert o.tok[0].tolist() == tok_x, (t, o.tok)
        assert o.lu[0].tolist() == lu_x, (t, o.lu)
        assert int(m[0]) == m_x, t
        assert int(o.t[0]) == t + 1
        pt = [-1] * C
        for s, p in enumerate(tok_x):
            if p >= 0:
                pt[p] = s
        assert o.pt[0].tolist() == pt, t
        for s, p in enumerate(tok_x):
            if p >= 0:
                assert (o.dev[0, s] == host[0, p]).all(), (t, s)


def test_hand_trace(oracle_mod):
    run_hand_trace(oracle_mod.Oracle)


# --------------------------------------------------------------------- textbook LRU, k = 1

def run_textbook_k1(Oracle, lib_path=None, seeds=range(6)):
    for seed in seeds:
        rng = random.Random(seed)
        C, S = rng.choice([(6, 2), (10, 3), (16, 5), (40, 7)])
        E = 16
        host = _host(1, C, E, seed)
        o = Oracle(1, C, S, E, lib_path=lib_path)
        ref = TextbookLRU(S)
        for step in range(120):
            x = rng.randrange(C) if rng.random() < 0.5 else rng.randrange(max(1, C // 3))
            out, m, _ = o.resolve(host, E, np.array([[x]], dtype=np.int32))
            assert int(m[0]) == int(ref.access(x)), (seed, step)
            resident = {int(p) for p in o.tok[0] if p >= 0}
            assert resident == ref.resident(), (seed, step)
            assert (o.dev[0, out[0, 0]] == host[0, x]).all()


def test_textbook_lru_k1(oracle_mod):
    run_textbook_k1(oracle_mod.Oracle)


# --------------------------------------------------------------------- recency-list LRU

def compare_with_list_model(o, ref, host, sel_rows, E):
    for t, sel in enumerate(sel_rows):
        out, m, _ = o.resolve(host, E, np.array([sel], dtype=np.int32))
        rout, rm, _ = ref.call(list(sel))
        assert out[0].tolist() == rout, (t, sel)
        assert int(m[0]) == rm, (t, sel)
        assert o.pt[0].tolist() == ref.page_table(), t
        assert o.tok[0].tolist() == ref.pos_in, t
        assert o.lu[0].tolist() == ref.touched, t
        # the stamp order the oracle keeps is the model's recency list
        lu = o.lu[0]
        assert sorted(range(ref.S), key=lambda s: (lu[s], s)) == ref.order, t
        dev = o.dev[0]
        for s, p in enumerate(ref.pos_in):
            if p >= 0:
                assert (dev[s] == host[0, p]).all(), (t, s)


def run_list_model_random(Oracle, lib_path=None, seeds=range(8), steps=40):
    for seed in seeds:
        rng = random.Random(100 + seed)
        C = rng.choice([8, 12, 24, 64])
        S = rng.choice([2, 3, 5, 8])
        k = rng.randint(1, min(S, C))
        E = 16
        host = _host(1, C, E, seed)
        o = Oracle(1, C, S, E, lib_path=lib_path)
        ref = RecencyListLRU(C, S)
        rows = []
        prev = rng.sample(range(C), k)
        for _ in range(steps):
            keep = rng.sample(prev, rng.randint(0, k))
            rest = [p for p in range(C) if p not in keep]
            row = keep + rng.sample(rest, k - len(keep))
            rng.shuffle(row)
            rows.append(row)
            prev = row
        compare_with_list_model(o, ref, host, rows, E)


def test_recency_list_model_random(oracle_mod):
    run_list_model_random(oracle_mod.Oracle)


def test_recency_list_model_exhaustive(oracle_mod):
    """Every sequence of three 2-subsets of 5 positions, S = 3 (and 1-subsets, S = 2)."""
    E = 8
    for C, S, k, T in ((5, 3, 2, 3), (4, 2, 1, 4)):
        host = _host(1, C, E, 7)
        subsets = list(itertools.combinations(range(C), k))
        for seq in itertools.product(subsets, repeat=T):
            o = oracle_mod.Oracle(1, C, S, E)
            ref = RecencyListLRU(C, S)
            compare_with_list_model(o, ref, host, [list(r) for r in seq], E)


# --------------------------------------------------------------------- closed forms

def test_cold_start_closed_form(oracle_mod):
    """From empty: every selected position misses; slot i holds the i-th smallest."""
    rng = np.random.default_rng(3)
    for C, S, k in ((64, 16, 16), (100, 40, 17), (4096, 512, 256)):
        o = oracle_mod.Oracle(1, C, S, 8)
        host = _host(1, C, 8)
        sel = rng.choice(C, size=k, replace=False).astype(np.int32)
        out, m, _ = o.resolve(host, 8, sel[None])
        assert int(m[0]) == k
        srt = np.sort(sel)
        assert o.tok[0, :k].tolist() == srt.tolist()
        assert (o.tok[0, k:] == -1).all()
        assert (o.lu[0, :k] == 0).all() and (o.lu[0, k:] == -1).all()
        assert out[0].tolist() == np.searchsorted(srt, sel).tolist()


def test_compulsory_misses_only_when_cache_holds_everything(oracle_mod, tg):
    """S >= C: the total miss count is the number of distinct positions ever selected."""
    for seed in range(4):
        C, S, k = 96, 96, 12
        sel = tg.raw_trace(2, C, k, 40, 70, 1.1, seed=seed)
        o = oracle_mod.Oracle(2, C, S, 8)
        host = _host(2, C, 8, seed)
        total = np.zeros(2, dtype=np.int64)
        for t in range(sel.shape[0]):
            _, m, _ = o.resolve(host, 8, sel[t])
            total += m
        for b in range(2):
            assert total[b] == len(np.unique(sel[:, b, :]))


def test_slots_equal_k_closed_form(oracle_mod, tg):
    """S = k: a call misses exactly the positions not selected in the previous call."""
    C, k = 500, 32
    sel = tg.raw_trace(3, C, k, 30, 60, 1.1, seed=5)
    o = oracle_mod.Oracle(3, C, k, 8)
    host = _host(3, C, 8)
    for t in range(sel.shape[0]):
        _, m, _ = o.resolve(host, 8, sel[t])
        for b in range(3):
            if t == 0:
                assert m[b] == k
            else:
                assert m[b] == len(set(sel[t, b]) - set(sel[t - 1, b]))


def test_miss_bound_of_locality_traces(oracle_mod, tg):
    """Any S >= k: m_t <= |S_t minus S_(t-1)| <= k - floor(keep * k / 100)."""
    for S in (64, 100, 400):
        C, k, keep = 2000, 64, 85
        sel = tg.raw_trace(2, C, k, 40, keep, 1.1, seed=S)
        o = oracle_mod.Oracle(2, C, S, 8)
        host = _host(2, C, 8)
        bound = k - (keep * k) // 100
        for t in range(sel.shape[0]):
            _, m, _ = o.resolve(host, 8, sel[t])
            if t > 0:
                for b in range(2):
                    fresh = len(set(sel[t, b]) - set(sel[t - 1, b]))
                    assert m[b] <= fresh <= bound


# --------------------------------------------------------------------- special inputs

def test_repeat_selection_costs_nothing(oracle_mod):
    rng = np.random.default_rng(9)
    o = oracle_mod.Oracle(1, 300, 40, 8)
    host = _host(1, 300, 8)
    sel = rng.choice(300, size=30, replace=False).astype(np.int32)[None]
    o.resolve(host, 8, sel)
    for _ in range(3):
        out, m, _ = o.resolve(host, 8, rng.permutation(sel[0])[None])
        assert m[0] == 0


def run_padding_range_and_duplicates(Oracle, lib_path=None, ERR_RANGE=1, ERR_DUP=2):
    C, S, E = 16, 4, 8
    host = _host(1, C, E)
    o = Oracle(1, C, S, E, lib_path=lib_path)
    out, m, st = o.resolve(host, E, np.array([[3, -1, 3, 99]], dtype=np.int32))
    assert st == ERR_RANGE | ERR_DUP
    assert m[0] == 1                      # position 3 counts once
    assert out[0].tolist() == [0, -1, 0, -1]
    assert o.tok[0].tolist() == [3, -1, -1, -1]
    assert (o.dev[0, 0] == host[0, 3]).all()
    out, m, st = o.resolve(host, E, np.array([[-5, 3, 4, -1]], dtype=np.int32))
    assert st == 0 and m[0] == 1
    assert out[0].tolist() == [-1, 0, 1, -1]
    assert o.lu[0].tolist() == [1, 1, -1, -1]


def test_padding_range_and_duplicates(oracle_mod):
    run_padding_range_and_duplicates(oracle_mod.Oracle, None, oracle_mod.ERR_RANGE,
                                     oracle_mod.ERR_DUP)


def test_permutation_invariance(oracle_mod, tg):
    """Permuting a row permutes the output and leaves the state unchanged."""
    C, S, k = 3000, 200, 96
    sel = tg.raw_trace(1, C, k, 20, 80, 1.1, seed=11)
    host = _host(1, C, 8)
    a = oracle_mod.Oracle(1, C, S, 8)
    b = oracle_mod.Oracle(1, C, S, 8)
    rng = np.random.default_rng(0)
    for t in range(sel.shape[0]):
        perm = rng.permutation(k)
        oa, ma, _ = a.resolve(host, 8, sel[t])
        ob, mb, _ = b.resolve(host, 8, sel[t][:, perm])
        assert (oa[:, perm] == ob).all() and (ma == mb).all()
        for name in ("pt", "tok", "lu", "t", "dev"):
            assert (getattr(a, name) == getattr(b, name)).all()


# --------------------------------------------------------------------- invariants on the workloads

def check_invariants(o, host, sel, out, m, t, k):
    B = sel.shape[0]
    pt, tok, lu, dev = o.pt, o.tok, o.lu, o.dev
    for b in range(B):
        s_out = out[b]
        assert ((s_out >= 0) & (s_out < o.S)).all()
        assert len(np.unique(s_out)) == k                 # distinct rows -> distinct slots
        hits = k - int(m[b])
        assert hits >= 0
        # every selected position is resident, through the page table
        assert (pt[b, sel[b]] == s_out).all()
        # pt and tok are mutually inverse; at most S positions mapped
        mapped = np.nonzero(pt[b] >= 0)[0]
        assert len(mapped) <= o.S
        assert (tok[b, pt[b, mapped]] == mapped).all()
        occ = np.nonzero(tok[b] >= 0)[0]
        assert len(occ) == len(mapped)
        assert (pt[b, tok[b, occ]] == occ).all()
        # stamps: slots used now carry t; others are older
        assert (lu[b, s_out] == t).all()
        assert (lu[b] <= t).all()
        # exactness: the consumer view and every occupied slot equal the host rows
        assert (dev[b, s_out] == host[b, sel[b]]).all()
        assert (dev[b, occ] == host[b, tok[b, occ]]).all()


@pytest.mark.parametrize("name,B,T", [("tiny", 1, 64), ("dsa", 2, 256), ("long", 1, 64),
                                      ("quest", 1, 40)])
def test_invariants_on_workloads(oracle_mod, tg, name, B, T):
    w = tg.WORKLOADS[name]
    sel = tg.trace(w, T=T, B=B)
    host = tg.fill_kv_array(w, B=B)
    o = oracle_mod.Oracle(B, w.C, w.S, w.E)
    bound = w.k - (w.keep_pct * w.k) // 100
    for t in range(T):
        out, m, st = o.resolve(host, w.E, sel[t])
        assert st == 0
        if t == 0:
            assert (m == w.k).all()
        else:
            assert (m <= bound).all()
        if t % 8 == 0 or t == T - 1:
            check_invariants(o, host, sel[t], out, m, t, w.k)


def test_invariants_sweep_and_trend(oracle_mod, tg):
    """Sweep points at B = 1 (fewer steps): invariants, and fewer misses with more slots."""
    T = 24
    totals = {}
    for keep in (50, 80, 95):
        for S in (2048, 4096, 6144):
            w = tg.sweep_workload(S, keep)
            sel = tg.trace(w, T=T, B=1)
            host = tg.fill_kv_array(w, B=1)
            o = oracle_mod.Oracle(1, w.C, S, w.E)
            tot = 0
            for t in range(T):
                out, m, _ = o.resolve(host, w.E, sel[t])
                tot += int(m.sum())
                if t in (0, T - 1):
                    check_invariants(o, host, sel[t], out, m, t, w.k)
            totals[(S, keep)] = tot
        # blog commentary, section three (figure 3): more slots, fewer misses
        assert totals[(2048, keep)] >= totals[(4096, keep)] >= totals[(6144, keep)]


def test_noio_trace_is_all_hits_after_first_call(oracle_mod, tg):
    w = tg.noio_workload(2048)
    sel = tg.trace(w, T=6, B=2)
    o = oracle_mod.Oracle(2, w.C, w.S, 16)
    host = np.zeros((2, w.C, 16), dtype=np.uint8)
    for t in range(6):
        _, m, _ = o.resolve(host, 16, sel[t])
        assert (m == (w.k if t == 0 else 0)).all()


# --------------------------------------------------------------------- decode-time append

def run_append(Oracle, lib_path=None, ERR_RANGE=1):
    """An appended entry is part of the host history (a later miss fetches it), and a
    rewrite of a resident entry reaches its slot at once (the consumer view stays exact)."""
    C, S, E = 32, 4, 16
    host = _host(1, C, E, 5)
    o = Oracle(1, C, S, E, lib_path=lib_path)
    new = np.full((1, E), 0xAB, dtype=np.uint8)
    assert o.append(host, [30], new) == 0           # not resident: host only
    assert (host[0, 30] == 0xAB).all()
    out, m, _ = o.resolve(host, E, np.array([[30, 2]], dtype=np.int32))
    assert m[0] == 2 and (o.dev[0, out[0, 0]] == 0xAB).all()
    new2 = np.full((1, E), 0x5C, dtype=np.uint8)
    state = (o.pt.copy(), o.tok.copy(), o.lu.copy(), o.t.copy())
    assert o.append(host, [2], new2) == 0            # resident: host and slot
    assert (host[0, 2] == 0x5C).all() and (o.dev[0, out[0, 1]] == 0x5C).all()
    for a, b_ in zip(state, (o.pt, o.tok, o.lu, o.t)):
        assert (a == b_).all()                      # replacement state untouched
    out2, m2, _ = o.resolve(host, E, np.array([[2, 30]], dtype=np.int32))
    assert m2[0] == 0 and (o.dev[0, out2[0, 0]] == 0x5C).all()
    assert o.append(host, [-1], new) == 0            # no new entry
    assert o.append(host, [C], new) == ERR_RANGE


def test_append_joins_the_history_and_keeps_the_cache_exact(oracle_mod):
    run_append(oracle_mod.Oracle, None, oracle_mod.ERR_RANGE)


# --------------------------------------------------------------------- replacement policies
# LRU is the method's policy; FIFO and RANDOM are the locality-blind comparisons of the
# blog commentary's Fig. 3 discussion (the pages name neither; both are read as the
# plainest policy of their kind).

LRU, FIFO, RANDOM = 0, 1, 2

# The textbook reference string of Belady's anomaly, one access per call.
BELADY = [1, 2, 3, 4, 1, 2, 5, 1, 2, 3, 4, 5]


def _calls(o, host, rows):
    outs, misses = [], []
    for sel in rows:
        out, m, _ = o.resolve(host, host.shape[2], np.asarray(sel, dtype=np.int32).reshape(o.R, -1))
        outs.append(out)
        misses.append(m)
    return outs, misses


def run_policies(Oracle, lib_path=None):
    E = 16
    # (1) Belady's string: FIFO faults 9 times with 3 frames and 10 with 4; LRU 10 and 8
    for policy, S, faults in ((FIFO, 3, 9), (FIFO, 4, 10), (LRU, 3, 10), (LRU, 4, 8)):
        o = Oracle(1, 8, S, E, lib_path=lib_path)
        o.set_policy(policy)
        _, m = _calls(o, _host(1, 8, E), [[x] for x in BELADY])
        assert int(np.sum(m)) == faults, (policy, S)
    # (2) FIFO against a textbook FIFO queue on random single-access traces; the stamp of
    #     every occupied slot is the call that filled it
    for seed in range(3):
        rng = random.Random(seed)
        C, S = rng.choice([(10, 3), (16, 5), (40, 7)])
        host = _host(1, C, E, seed)
        o = Oracle(1, C, S, E, lib_path=lib_path)
        o.set_policy(FIFO)
        ref = TextbookFIFO(S)
        filled = [-1] * S
        for t in range(150):
            x = rng.randrange(C) if rng.random() < 0.5 else rng.randrange(max(1, C // 3))
            out, m, _ = o.resolve(host, E, np.array([[x]], dtype=np.int32))
            assert int(m[0]) == int(ref.access(x)), (seed, t)
            if m[0]:
                filled[out[0, 0]] = t
            assert {int(p) for p in o.tok[0] if p >= 0} == ref.resident(), (seed, t)
            assert o.lu[0].tolist() == filled, (seed, t)
            assert (o.dev[0, out[0, 0]] == host[0, x]).all()
    # (3) RANDOM: the victims of every call are the non-hit slots with the smallest
    #     (key, slot), keys from SplitMix64 as published, request numbers honoured
    seed = 0xC0FFEE
    C, S, k, R = 64, 12, 4, 3
    host = _host(R, C, E, 3)
    o = Oracle(R, C, S, E, lib_path=lib_path)
    o.set_policy(RANDOM, seed)
    ids = [5, 0, 1 << 19]
    o.set_request_ids(ids)
    rng = np.random.default_rng(4)
    for t in range(60):
        sel = np.stack([rng.choice(C if t % 3 else 20, size=k, replace=False) for _ in range(R)]).astype(np.int32)
        tok0 = o.tok.copy()
        out, m, _ = o.resolve(host, E, sel)
        for b in range(R):
            hit = {int(s) for s in range(S) if tok0[b, s] >= 0 and tok0[b, s] in set(sel[b].tolist())}
            stream = splitmix64(seed, ids[b])
            cand = sorted((splitmix64(stream, (t << 16) + s) >> 32, s) for s in range(S) if s not in hit)
            missed = sorted({int(p) for p in sel[b]} - {int(tok0[b, s]) for s in hit})
            assert int(m[b]) == len(missed)
            for p, (_, v) in zip(missed, cand):
                assert int(o.pt[b, p]) == v and int(o.tok[b, v]) == p, (t, b)
            for j, p in enumerate(sel[b]):
                assert (o.dev[b, out[b, j]] == host[b, p]).all()
    # (4) a loop over S + 1 positions: LRU and FIFO miss on every call (the textbook
    #     pathology of recency and arrival order), RANDOM keeps some of the loop
    S = 6
    loop = [[x % (S + 1)] for x in range(20 * (S + 1))]
    for policy, none_hit in ((LRU, True), (FIFO, True), (RANDOM, False)):
        o = Oracle(1, S + 1, S, E, lib_path=lib_path)
        o.set_policy(policy, 9)
        _, m = _calls(o, _host(1, S + 1, E), loop)
        hits = len(loop) - int(np.sum(m))
        assert (hits == 0) == none_hit, (policy, hits)


def test_replacement_policies(oracle_mod):
    run_policies(oracle_mod.Oracle)


def test_splitmix64_published_outputs(oracle_mod):
    """SplitMix64's published outputs for seeds 0 and 1234567, for the test's model and
    for the oracle's generator."""
    want = {0: [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F],
            1234567: [6457827717110365317, 3203168211198807973, 9817491932198370423,
                      4593380528125082431, 16408922859458223821]}
    for seed, outs in want.items():
        for n, v in enumerate(outs):
            assert splitmix64(seed, n) == v
            assert oracle_mod.splitmix64(seed, n) == v
    assert oracle_mod.random_key(7, 3, 11, 5) == splitmix64(splitmix64(7, 3), (11 << 16) + 5) >> 32


def test_random_victims_are_uniform(oracle_mod):
    """With every call a miss on a full cache, each of the S slots is the victim about
    equally often (chi-square, 7 degrees of freedom, below the 0.1 % quantile 24.3)."""
    S, n = 8, 4000
    o = oracle_mod.Oracle(1, n + S, S, 16)
    o.set_policy(RANDOM, 12345)
    host = _host(1, n + S, 16)
    counts = np.zeros(S)
    for x in range(n + S):
        out, m, _ = o.resolve(host, 16, np.array([[x]], dtype=np.int32))
        assert m[0] == 1
        if x >= S:
            counts[out[0, 0]] += 1
    chi2 = float(((counts - n / S) ** 2 / (n / S)).sum())
    assert chi2 < 24.3, counts
