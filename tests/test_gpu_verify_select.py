"""Verify with the Top-K selection fused into the criticality pass: the same outputs, scores and
selection as the separate verify and select calls (bit-exact: the same arithmetic and the same row
selection), and a selection the oracle's Top-K reproduces from the GPU's scores."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import (KVCache, SpecRound, binding, ssd_select_topk, ssd_status,
                                                 ssd_verify_attn, ssd_verify_select)
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _both(w, ks=None, k_max=None, expect_status=0):
    _gpu.lib()
    spec = w.spec
    kv = KVCache.from_workload(w)
    scale = _gpu.scale_of(spec)
    ks = w.k_per_req if ks is None else ks
    k_max = int(ks.max()) if k_max is None else k_max
    f = ssd_verify_select(kv, w.q_verify, spec.n_cand, scale, ks, k_max)
    torch.cuda.synchronize()
    assert ssd_status() == expect_status
    u = ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale)
    ui, uc = ssd_select_topk(u["scores"], kv.seq_lens, ks, k_max, spec.h_kv, max_len=kv.max_seq_len)
    torch.cuda.synchronize()
    assert ssd_status() == expect_status
    for name in ("out", "lse", "scores"):
        assert torch.equal(f[name], u[name]), name
    assert torch.equal(f["cnt"], uc)
    assert torch.equal(f["idx"], ui)
    return kv, f


CASES = [
    # (B, lens, h_q, h_kv, d, n_cand, page_size)
    (3, [700, 129, 5000], 32, 8, 128, 5, 16),   # one and three 2048-token score blocks per row
    (2, [4097, 2048], 32, 8, 128, 7, 16),       # exact block multiple and one token past it
    (2, [1111, 2222], 8, 2, 64, 3, 64),         # d = 64 (mma.sync verify)
    (1, [5], 4, 2, 128, 5, 16),                 # L = n_cand
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}-L{'_'.join(map(str, c[1]))}-d{c[4]}-nc{c[5]}")
def test_fused_matches_separate_calls(case):
    B, lens, h_q, h_kv, d, nc, ps = case
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="vsel", batch=B, h_q=h_q, h_kv=h_kv, d=d, k=nc - 1, page_size=ps)
    w = W.make_workload(spec, seed=31 + sum(lens), device=DEV, lengths=lens, spare_pages=3)
    kv, f = _both(w)
    # The selection is the oracle's Top-K of the same fp32 scores.
    S = f["scores"].cpu().numpy()
    oi, oc = oracle.topk(S.reshape(-1, S.shape[-1]), kv.seq_lens.cpu().numpy(), w.k_per_req.cpu().numpy(),
                         f["idx"].shape[1], rows_per_group=h_kv)
    np.testing.assert_array_equal(f["idx"].cpu().numpy(), oi)
    np.testing.assert_array_equal(f["cnt"].cpu().numpy(), oc)


def test_fused_tiny_fp32_and_select_all():
    """The fp32 path; K = L keeps every token."""
    w = W.make_workload(W.SPECS["tiny"], device=DEV)
    _both(w)
    _both(w, ks=w.seq_lens.clone())


def test_fused_k_over_kmax_faults_and_truncates():
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="vsel_k", batch=2)
    w = W.make_workload(spec, seed=41, device=DEV, lengths=[3000, 900])
    ks = torch.tensor([200, 40], dtype=torch.int32, device=DEV)
    _, f = _both(w, ks=ks, k_max=100, expect_status=binding.FAULT_KMAX)
    assert f["cnt"].cpu().view(2, -1)[0].tolist() == [100] * spec.h_kv
    assert f["cnt"].cpu().view(2, -1)[1].tolist() == [40] * spec.h_kv


def test_fused_repeated_calls_and_shapes():
    """The arrival counters return to zero: consecutive calls of different shapes on one workspace."""
    _gpu.lib()
    ws = binding.Workspace()
    for seed, lens in ((51, [3000, 100, 4500]), (52, [64, 2049]), (53, [3000, 100, 4500])):
        spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="vsel_r", batch=len(lens))
        w = W.make_workload(spec, seed=seed, device=DEV, lengths=lens)
        kv = KVCache.from_workload(w)
        k_max = int(w.k_per_req.max())
        scale = _gpu.scale_of(spec)
        f = ssd_verify_select(kv, w.q_verify, spec.n_cand, scale, w.k_per_req, k_max, workspace=ws)
        u = ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale, workspace=ws)
        ui, uc = ssd_select_topk(u["scores"], kv.seq_lens, w.k_per_req, k_max, spec.h_kv, max_len=kv.max_seq_len)
        torch.cuda.synchronize()
        assert ssd_status() == 0
        assert torch.equal(f["idx"], ui) and torch.equal(f["cnt"], uc)


def test_fused_round_full_size_and_graph():
    """The full-size Qwen3-8B round with the fused selection equals the separate one, eagerly and as
    a replayed CUDA graph."""
    _gpu.lib()
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, device=DEV)
    k_max = int(w.k_per_req.max())
    scale = _gpu.scale_of(spec)
    a = SpecRound(KVCache.from_workload(w), spec.h_q, spec.n_cand, k_max, scale)
    b = SpecRound(KVCache.from_workload(w), spec.h_q, spec.n_cand, k_max, scale)
    oa = torch.empty((spec.k, spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=DEV)
    ob = torch.empty_like(oa)
    a.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=oa)
    b.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=ob, fused_select=True)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(a.idx, b.idx) and torch.equal(a.cnt, b.cnt) and torch.equal(oa, ob)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        b.idx.zero_()
        ob.zero_()
        with torch.cuda.graph(g, stream=s):
            b.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=ob, fused_select=True)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(a.idx, b.idx) and torch.equal(oa, ob)
