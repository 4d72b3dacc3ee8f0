"""Planted mistakes: each edit below breaks the oracle in a plausible way, and the
pins of test_oracle_pins must catch every one of them.

The mistakes are planted in temporary copies of the oracle's C source, compiled on
the CPU; the oracle itself is never modified.
"""
import os

import pytest

from tests import test_oracle_attend as attend_pins
from tests import test_oracle_pins as pins
from tests import test_pool_plan as pool_pins

MUTANTS = {
    "tie_break_reversed": ("return (x->slot > y->slot) - (x->slot < y->slot);",
                           "return (x->slot < y->slot) - (x->slot > y->slot);"),
    "misses_descending": ("return (x > y) - (x < y);", "return (x < y) - (x > y);"),
    "hits_evictable": ("        if (hit[s]) continue;\n", ""),
    "no_unmap": ("if (tok[v] >= 0) pt[tok[v]] = -1;", ""),
    "hits_not_stamped": ("for (int s = 0; s < S; ++s) if (hit[s]) lu[s] = t;", ""),
    "victims_not_stamped": ("for (int i = 0; i < m; ++i) lu[V[i].slot] = t;", ""),
    "stamp_off_by_one": ("if (hit[s]) lu[s] = t;", "if (hit[s]) lu[s] = t + 1;"),
    "wrong_row_fetched": ("host_b + (size_t)P[i] * host_stride", "host_b + (size_t)v * host_stride"),
    "most_recent_victim": ("int32_t v = V[i].slot;", "int32_t v = V[nv - 1 - i].slot;"),
    "step_not_advanced": ("o->t[b] = t + 1;", "o->t[b] = t;"),
    "duplicate_miss_counted_twice": ("*miss_b = m;", "*miss_b = np;"),
    "append_skips_resident_slot": ("if (s >= 0) memcpy(o->dev + ((size_t)b * o->S + s) * o->E, row, (size_t)o->E);", ""),
    "most_recent_first_order": ("if (x->key != y->key) return (x->key > y->key) - (x->key < y->key);",
                                "if (x->key != y->key) return (x->key < y->key) - (x->key > y->key);"),
    "attend_scale_block_of_64": ("memcpy(&sc, row + 512 + 4 * (d / 128), 4);", "memcpy(&sc, row + 512 + 4 * ((d / 64) & 3), 4);"),
    "attend_rope_dropped": ("K[(size_t)j * 576 + 512 + d] = orc_bf16(h);", "K[(size_t)j * 576 + 512 + d] = 0.0;"),
    "attend_lse_without_max": ("lse[h] = mx + log(l);", "lse[h] = log(l);"),
    "attend_padding_clamped": ("const int32_t sl = out_b[j];", "const int32_t sl = out_b[j] < 0 ? 0 : out_b[j];"),
    "e4m3_bias_8": ("else v = ldexp(1.0 + (double)m / 8.0, e - 7);", "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal_scale": ("if (e == 0) v = ldexp((double)m / 8.0, -6);", "if (e == 0) v = ldexp((double)m / 8.0, -7);"),
    "length_ignored_in_range": ("if (p >= lim) { status |= ORC_ERR_RANGE; continue; }",
                                "if (p >= C) { status |= ORC_ERR_RANGE; continue; }"),
    "reset_keeps_call_counter": ("    o->t[b] = 0;\n    memset(", "    memset("),
    "fifo_restamps_hits": ("if (o->policy != ORC_POLICY_FIFO)\n", "if (1)\n"),
    "random_key_low_bits": ("+ (uint64_t)s) >> 32);", "+ (uint64_t)s));"),
    "random_key_ignores_request": ("orc_random_key(o->seed, o->rid[b], t, s)", "orc_random_key(o->seed, b, t, s)"),
    "random_counter_swapped": ("((uint64_t)(uint32_t)t << 16) + (uint64_t)s", "((uint64_t)(uint32_t)s << 16) + (uint64_t)t"),
    "random_policy_uses_stamps": ("o->policy == ORC_POLICY_RANDOM ?", "o->policy == -7 ?"),
}


def _pin_suite(Oracle, path):
    pool_pins.run_length_limit(Oracle, path)
    attend_pins.run_attend(Oracle, path)
    pins.run_policies(Oracle, path)
    pins.run_append(Oracle, path)
    pins.run_hand_trace(Oracle, path)
    pins.run_textbook_k1(Oracle, path, seeds=range(3))
    pins.run_list_model_random(Oracle, path, seeds=range(4), steps=25)
    pins.run_padding_range_and_duplicates(Oracle, path)


def test_unmutated_copy_passes(oracle_mod, tmp_path):
    src = open(oracle_mod.SRC).read()
    p = tmp_path / "o.c"
    p.write_text(src)
    so = oracle_mod.compile_oracle(str(p), str(tmp_path / "o.so"))
    _pin_suite(oracle_mod.Oracle, so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle_mod.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    p = tmp_path / f"{name}.c"
    p.write_text(src.replace(old, new))
    so = oracle_mod.compile_oracle(str(p), str(tmp_path / f"{name}.so"))
    with pytest.raises(AssertionError):
        _pin_suite(oracle_mod.Oracle, so)
