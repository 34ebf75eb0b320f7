"""Planted mistakes in the CPU oracle must be caught by the pins.

Each mutant is a one-line change to a copy of the oracle source (compiled with gcc into a
temporary directory); the pin battery of ``tests/_pins.py`` has to fail on it.  Nothing here
touches a GPU.
"""

import os
import subprocess

import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("int last = L - c->n_c + i; /* R1 */", "int last = L - c->n_c + i - 1;"),
    "causal_sees_all": ("int last = L - c->n_c + i; /* R1 */", "int last = L - 1;"),
    "gqa_head_strided": ("int h = g * G + hl; /* query head h reads KV head h / G */",
                         "int h = hl * kv->h_kv + g;"),
    "scale_dropped": ("*s = scale * acc;", "*s = acc;"),
    "crit_first_candidate_only": ("if (crit) crit[t] += p[t];", "if (crit && i == 0) crit[t] += p[t];"),
    "softmax_no_max_shift_in_p": ("double p = exp(s_buf[j] - m) / z;", "double p = exp(s_buf[j]) / z;"),
    "value_uses_key": ("int rc = orc_row(kv, b, 1, g, tokens[j], &off);",
                       "int rc = orc_row(kv, b, 0, g, tokens[j], &off);"),
    "topk_ties_to_higher_index": ("return (x->i > y->i) - (x->i < y->i);", "return (x->i < y->i) - (x->i > y->i);"),
    "topk_unsorted_output": ("qsort(out, (size_t)k, sizeof(int32_t), orc_cmp_int);", ";"),
    "maxpool_first_not_max": ("m = src[t] > m ? src[t] : m;", "m = (t == j * block) ? src[t] : m;"),
    "union_mask_bit_wrong": ("umask[(int64_t)u * umax + m - 1] |= 1u << all[j].cand;",
                             "umask[(int64_t)u * umax + m - 1] |= 1u;"),
    "block_attn_no_causal": ("int last = L - c->n_c + i, n = 0;", "int last = L - 1, n = 0;"),
    "page_slot_wrong": ("(t % kv->page_size)) * kv->d;", "(t / kv->page_size) % kv->page_size) * kv->d;"),
    "append_slot_shifted": ("* page_size + t % page_size) * row_bytes;", "* page_size + (t + 1) % page_size) * row_bytes;"),
    "append_k_v_swapped": ("(which ? v_new : k_new)", "(which ? k_new : v_new)"),
    "phase_ties_to_highest": ("if (counts[o] < counts[best]) best = o;", "if (counts[o] <= counts[best]) best = o;"),
    "phase_verify_is_first": ("== n_buckets - 1);", "== 0);"),
    "topp_strict_reach": ("while (k < n && acc < target) acc += (double)pairs[k++].v;",
                          "while (k < n && acc <= target) acc += (double)pairs[k++].v;"),
    "topp_no_cap": ("kout[r] = k < k_max ? k : k_max;", "kout[r] = k;"),
    "combine_weight_unnormalised": ("const double w = exp((double)lp[j] - total);",
                                    "const double w = exp((double)lp[j] - m);"),
    "combine_lse_is_max": ("    lse[r] = total;", "    lse[r] = m;"),
    "advance_no_range_check": ("if (v >= 0 && v <= max_seq_len) seq_lens[b] = (int32_t)v;", "seq_lens[b] = (int32_t)v;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/present"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", str(so), str(path), "-lm"],
                   check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, name, old, new)
    failures = []
    oracle._use_library(so)
    try:
        for pin in _pins.ALL_PINS:
            try:
                pin(oracle)
            except (AssertionError, ValueError) as e:  # a pin failed, or the oracle rejected its input
                failures.append((pin.__name__, type(e).__name__))
    finally:
        oracle._use_library(None)
    assert failures, f"no pin caught mutant {name}"
