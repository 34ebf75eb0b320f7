"""Byte accounting used by the benchmark, pinned to the figure the SparseSpec page prints."""

import os

from sparse_self_speculative_verify_gb300 import metrics as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes_qwen3_8b.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            vals[k] = int(v)
    return vals


def test_kv_bytes_per_step_matches_page():
    g = _golden()
    per_tok = M.kv_bytes_per_token(g["h_kv"], g["d"], g["elem_bytes"], layers=g["layers"])
    assert per_tok * g["tokens"] == g["total_bytes"]
    assert g["total_bytes"] == 18 * 2 ** 20


def test_round_bytes_decompose():
    lens = [2048, 8192, 5000]
    ks = [103, 410, 250]
    v = M.verify_kv_bytes(lens, 8, 128, 2)
    assert v == sum(lens) * 8 * 512
    d = M.draft_kv_bytes(ks, lens, 8, 128, 2)
    assert d == sum(ks) * 8 * 512
    assert M.round_kv_bytes(lens, ks, 8, 128, 2, 4) == v + 4 * d


def test_verify_flops_counts_visible_pairs():
    # One request, L = 6, n_cand = 3: candidates see 4, 5 and 6 tokens.
    assert M.verify_flops([6], h_q=2, d=4, n_cand=3) == (4 + 5 + 6) * 2 * 4 * 4
