"""Sparse draft attention on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import KVCache, ssd_draft_attn, ssd_status, ssd_verify_attn
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _draft(w, idx, cnt, q=None):
    _gpu.lib()
    kv = KVCache.from_workload(w)
    q = w.q_draft[0] if q is None else q
    r = ssd_draft_attn(kv, q, idx.to(DEV), cnt.to(DEV), _gpu.scale_of(w.spec))
    torch.cuda.synchronize()
    assert ssd_status() == 0
    return r


def _check(w, r, idx, cnt, reqs=None, q=None):
    kv_h, reqs = _gpu.host_subset(w, reqs)
    q = (w.q_draft[0] if q is None else q).cpu()[reqs]
    ref = oracle.draft(kv_h, q, idx[reqs], cnt[reqs], _gpu.scale_of(w.spec))
    _gpu.assert_out(r["out"].cpu().numpy()[reqs], ref["out"], "draft out")
    _gpu.assert_lse(r["lse"].cpu().numpy()[reqs], ref["lse"])


CASES = [
    # (spec name, overrides, lens, k per request, k_max)
    ("qwen3_8b", dict(batch=3), [2049, 700, 64], [103, 35, 64], 128),       # 1-2 chunks per unit
    ("qwen3_8b", dict(batch=2), [8192, 5000], [410, 250], 410),               # 7 chunks: last-arriver merge
    ("qwen3_8b", dict(batch=2, h_q=40), [3000, 1200], [150, 0], 150),         # G = 5, one empty list
    ("qwen3_8b", dict(batch=2, h_q=128, h_kv=8), [600, 1000], [30, 300], 300),  # G = 16
    ("qwen3_8b", dict(batch=2, d=64, page_size=32), [1000, 333], [65, 17], 65),
    ("tiny", dict(), [512, 512], [64, 64], 64),                               # fp32, d = 64
    ("tiny", dict(d=128, page_size=16, shuffled=True), [700, 129], [100, 7], 100),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{'_'.join(map(str, c[2]))}-k{c[4]}")
def test_draft_random_sets(case):
    name, over, lens, ks, k_max = case
    spec = W.scaled_spec(W.SPECS[name], name="d", **over)
    w = W.make_workload(spec, seed=31 + k_max, device=DEV, lengths=lens)
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), k_max, seed=k_max)
    _check(w, _draft(w, idx, cnt), idx, cnt)


# Lists of exactly four 64-row chunks (256), one row more (257), seventeen chunks (1025), fewer rows
# than one warp's 16 (15), G = 1 / 5 / 16, and pages of 8, 32 and 64 tokens (rows are gathered one
# token at a time, anywhere in a page).
GATHER_CASES = [
    (dict(batch=4, page_size=8), [4000, 3000, 2000, 600], [256, 257, 1025, 15], 1025),
    (dict(batch=2, page_size=64, h_q=8), [5000, 3000], [640, 63], 640),
    (dict(batch=2, page_size=32, h_q=40), [9000, 2500], [700, 128], 700),
    (dict(batch=2, h_q=128), [3000, 900], [513, 191], 513),
]


@pytest.mark.parametrize("case", GATHER_CASES, ids=lambda c: f"ps{c[0]['page_size'] if 'page_size' in c[0] else 16}-"
                         f"hq{c[0].get('h_q', 32)}-k{c[3]}")
def test_draft_gather_boundaries(case):
    over, lens, ks, k_max = case
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="dgb", **over)
    w = W.make_workload(spec, seed=61 + k_max, device=DEV, lengths=lens)
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), k_max, seed=k_max + 5)
    _check(w, _draft(w, idx, cnt), idx, cnt)


def test_draft_many_short_lists():
    """A batch of 1040 (request, KV head) lists of 5 to 44 rows: one chunk each, every unit's output
    written by its single chunk."""
    lens = [int(x) for x in np.random.default_rng(3).integers(100, 900, size=130)]
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="dmany", batch=130)
    w = W.make_workload(spec, seed=17, device=DEV, lengths=lens)
    ks = [max(1, L // 20) for L in lens]
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), max(ks), seed=4)
    _check(w, _draft(w, idx, cnt), idx, cnt)


def test_draft_repeat_calls_identical():
    """Consecutive calls reuse the workspace counters: results are bit-identical."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="rep", batch=2)
    w = W.make_workload(spec, seed=2, device=DEV, lengths=[8000, 4000])
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor([400, 200], dtype=torch.int32), 400, seed=3)
    a = _draft(w, idx, cnt)["out"].clone()
    b = _draft(w, idx, cnt)["out"]
    assert torch.equal(a, b)


def test_draft_workspace_reused_across_shapes():
    """One workspace serves calls of different shapes in turn: the counters of the second call sit
    where the first call left partial outputs, and each call clears them before its kernel."""
    from sparse_self_speculative_verify_gb300 import Workspace
    ws = Workspace()
    specs = [(W.scaled_spec(W.SPECS["qwen3_8b"], name="wsa", batch=3), [8192, 6000, 300], [410, 300, 20], 410),
             (W.scaled_spec(W.SPECS["qwen3_8b"], name="wsb", batch=2, h_q=40), [3000, 5000], [150, 250], 250)]
    for n, (spec, lens, ks, k_max) in enumerate(specs + specs[:1]):
        w = W.make_workload(spec, seed=40 + n % 2, device=DEV, lengths=lens)
        idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), k_max, seed=n % 2)
        r = ssd_draft_attn(KVCache.from_workload(w), w.q_draft[0], idx.to(DEV), cnt.to(DEV), _gpu.scale_of(spec),
                           workspace=ws)
        torch.cuda.synchronize()
        assert ssd_status() == 0
        _check(w, r, idx, cnt)


def test_draft_select_all_equals_verify_single_candidate():
    """With every index selected, the draft is dense single-query attention: it matches the GPU
    verify with n_cand = 1 on the same query (and the oracle)."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="all", batch=2, k=0)
    w = W.make_workload(spec, seed=5, device=DEV, lengths=[1500, 700])
    k_max = 1500
    idx = torch.full((2, spec.h_kv, k_max), -1, dtype=torch.int32)
    cnt = torch.zeros((2, spec.h_kv), dtype=torch.int32)
    for b, L in enumerate([1500, 700]):
        idx[b, :, :L] = torch.arange(L, dtype=torch.int32)
        cnt[b] = L
    q = w.q_verify[:, 0].contiguous()
    r = _draft(w, idx, cnt, q=q)
    v = ssd_verify_attn(KVCache.from_workload(w), w.q_verify, 1, _gpu.scale_of(spec))
    torch.cuda.synchronize()
    _gpu.assert_out(r["out"].cpu().numpy(), v["out"][:, 0].cpu().numpy(), "draft vs verify", tol=1e-3)
    _check(w, r, idx, cnt, q=q)


def test_draft_full_size_qwen3_8b():
    """Full-size Qwen3-8B shape with 5% random index sets; every output against the oracle."""
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, device=DEV)
    k_max = int(w.k_per_req.max())
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, w.k_per_req, k_max, seed=77)
    _check(w, _draft(w, idx, cnt), idx, cnt)
