"""A whole speculative round (verify -> select -> k drafts) on the full-size Qwen3-8B-shaped
workload, as the benchmark runs it, plus its CUDA-graph replay."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import KVCache, SpecRound, ssd_draft_attn, ssd_status
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _round(w):
    _gpu.lib()
    spec = w.spec
    kv = KVCache.from_workload(w)
    k_max = int(w.k_per_req.max())
    rnd = SpecRound(kv, spec.h_q, spec.n_cand, k_max, _gpu.scale_of(spec))
    outs = torch.empty((spec.k, spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=DEV)
    rnd.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=outs)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    return rnd, outs


def test_round_qwen3_8b_full_size():
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, device=DEV)
    rnd, outs = _round(w)
    reqs = [1, 17, 31]
    kv_h, reqs = _gpu.host_subset(w, reqs)
    scale = _gpu.scale_of(spec)
    ref = oracle.verify(kv_h, w.q_verify.cpu()[reqs], scale)
    _gpu.assert_out(rnd.out_v.cpu().numpy()[reqs], ref["out"], "verify out")
    lens = kv_h.seq_lens
    _gpu.assert_scores(rnd.scores.cpu().numpy()[reqs], ref["crit"], lens)
    # The GPU's selection (from its own scores) is a valid top-K of the oracle's scores.
    k_max = rnd.k_max
    idx = rnd.idx.view(spec.batch, spec.h_kv, k_max).cpu().numpy()[reqs].reshape(-1, k_max)
    cnt = rnd.cnt.view(spec.batch, spec.h_kv).cpu().numpy()[reqs].reshape(-1)
    kpr = w.k_per_req.cpu().numpy()[reqs]
    _gpu.assert_valid_topk(idx, cnt, ref["crit"].reshape(-1, ref["crit"].shape[-1]), kpr, lens, spec.h_kv)
    # Drafts on the oracle's selection (fp32 scores, oracle top-K) against the oracle drafts.
    S = ref["crit"].astype(np.float32)
    oidx, ocnt = oracle.topk(S.reshape(-1, S.shape[-1]), lens, kpr, k_max, rows_per_group=spec.h_kv)
    oidx = oidx.reshape(len(reqs), spec.h_kv, k_max)
    ocnt = ocnt.reshape(len(reqs), spec.h_kv)
    full_idx = torch.zeros((spec.batch, spec.h_kv, k_max), dtype=torch.int32)
    full_cnt = torch.zeros((spec.batch, spec.h_kv), dtype=torch.int32)
    full_idx[reqs] = torch.from_numpy(oidx)
    full_cnt[reqs] = torch.from_numpy(ocnt)
    kv = KVCache.from_workload(w)
    for j in range(spec.k):
        g = ssd_draft_attn(kv, w.q_draft[j], full_idx.to(DEV), full_cnt.to(DEV), scale)
        dref = oracle.draft(kv_h, w.q_draft[j].cpu()[reqs], oidx, ocnt, scale)
        torch.cuda.synchronize()
        _gpu.assert_out(g["out"].cpu().numpy()[reqs], dref["out"], f"draft {j}")


def test_round_b128_l8k_full_size():
    """The 128 x 8192, k = 6 workload as the benchmark's rounds run it.  On sampled requests: the
    verify output and scores against the oracle; the GPU selection bit-exact against the oracle's
    Top-K of the same (GPU) score tensor and a valid Top-K of the oracle's scores; then the round's
    six drafts (the first storing the row pack, the other five reading it, K = 410 on every unit)
    on the oracle's own selection, against the oracle drafts."""
    spec = W.SPECS["b128_l8k"]
    w = W.make_workload(spec, device=DEV)
    rnd, _ = _round(w)
    B, hkv, k_max = spec.batch, spec.h_kv, rnd.k_max
    reqs = [0, 77, 127]
    kv_h, reqs = _gpu.host_subset(w, reqs)
    scale = _gpu.scale_of(spec)
    lens = kv_h.seq_lens
    kpr = w.k_per_req.cpu().numpy()[reqs]
    ref = oracle.verify(kv_h, w.q_verify.cpu()[reqs], scale)
    _gpu.assert_out(rnd.out_v.cpu().numpy()[reqs], ref["out"], "verify out")
    _gpu.assert_lse(rnd.lse_v.cpu().numpy()[reqs], ref["lse"], "verify lse")
    _gpu.assert_scores(rnd.scores.cpu().numpy()[reqs], ref["crit"], lens)
    Sg = rnd.scores.cpu().numpy()[reqs]
    gidx, gcnt = oracle.topk(Sg.reshape(-1, Sg.shape[-1]), lens, kpr, k_max, rows_per_group=hkv)
    idx = rnd.idx.view(B, hkv, k_max).cpu().numpy()[reqs].reshape(-1, k_max)
    cnt = rnd.cnt.view(B, hkv).cpu().numpy()[reqs].reshape(-1)
    np.testing.assert_array_equal(idx, gidx)
    np.testing.assert_array_equal(cnt, gcnt)
    _gpu.assert_valid_topk(idx, cnt, ref["crit"].reshape(-1, ref["crit"].shape[-1]), kpr, lens, hkv)
    S = ref["crit"].astype(np.float32)
    oidx, ocnt = oracle.topk(S.reshape(-1, S.shape[-1]), lens, kpr, k_max, rows_per_group=hkv)
    oidx = oidx.reshape(len(reqs), hkv, k_max)
    ocnt = ocnt.reshape(len(reqs), hkv)
    sel_idx = rnd.idx.view(B, hkv, k_max).clone()
    sel_cnt = rnd.cnt.view(B, hkv).clone()
    sel_idx[reqs] = torch.from_numpy(oidx).to(DEV)
    sel_cnt[reqs] = torch.from_numpy(ocnt).to(DEV)
    rnd.set_selection(sel_idx, sel_cnt)
    outs = torch.empty((spec.k, B, spec.h_q, spec.d), dtype=torch.float32, device=DEV)
    for j in range(spec.k):
        rnd.draft(w.q_draft[j], out=outs[j])
    torch.cuda.synchronize()
    assert ssd_status() == 0
    for j in range(spec.k):
        dref = oracle.draft(kv_h, w.q_draft[j].cpu()[reqs], oidx, ocnt, scale)
        _gpu.assert_out(outs[j].cpu().numpy()[reqs], dref["out"], f"draft {j}")


def test_round_graph_replay_matches_eager():
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="graph", batch=4)
    w = W.make_workload(spec, seed=3, device=DEV, lengths=[2100, 4097, 300, 1000])
    rnd, outs = _round(w)
    eager = (rnd.out_v.clone(), rnd.scores.clone(), rnd.idx.clone(), outs.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        rnd.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=outs)  # warm-up on the capture stream
        torch.cuda.synchronize()
        rnd.out_v.zero_()
        outs.zero_()
        with torch.cuda.graph(g, stream=s):
            rnd.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=outs)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(rnd.out_v, eager[0])
    assert torch.equal(rnd.scores, eager[1])
    assert torch.equal(rnd.idx, eager[2])
    assert torch.equal(outs, eager[3])


def _oracle_topk_case(lengths, seed, select_all=False):
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="otk", batch=len(lengths))
    w = W.make_workload(spec, seed=seed, device=DEV, lengths=lengths)
    _gpu.lib()
    kv = KVCache.from_workload(w)
    scale = _gpu.scale_of(spec)
    kpr = w.seq_lens.clone() if select_all else w.k_per_req
    k_max = int(kpr.max())
    rnd = SpecRound(kv, spec.h_q, spec.n_cand, k_max, scale)
    qd = w.q_draft[0]
    r = rnd.draft_oracle_topk(qd, kpr)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    kv_h, _ = _gpu.host_subset(w)
    return spec, w, kv_h, scale, kpr.cpu().numpy(), k_max, r


def test_oracle_topk_draft_matches_oracle():
    """'Oracle top-k' draft: the draft query's own criticality (a verify with one candidate, which
    sees the whole cache) selects its tokens.  Dense output and scores against the oracle's, the
    selection bit-exact against the oracle's Top-K of the GPU's scores, the sparse output against
    the oracle draft on that selection."""
    spec, w, kv_h, scale, kpr, k_max, r = _oracle_topk_case([3000, 1029, 4500], 21)
    qd = w.q_draft[0].cpu()
    ref = oracle.verify(kv_h, qd[:, None], scale)
    lens = kv_h.seq_lens
    _gpu.assert_out(r["dense"].cpu().numpy(), ref["out"][:, 0], "dense")
    _gpu.assert_scores(r["scores"].cpu().numpy(), ref["crit"], lens)
    S = r["scores"].cpu().numpy()
    oidx, ocnt = oracle.topk(S.reshape(-1, S.shape[-1]), lens, kpr, k_max, rows_per_group=spec.h_kv)
    np.testing.assert_array_equal(r["idx"].cpu().numpy(), oidx)
    np.testing.assert_array_equal(r["cnt"].cpu().numpy(), ocnt)
    # The selection is also a valid Top-K of the oracle's own scores.
    _gpu.assert_valid_topk(oidx, ocnt, ref["crit"].reshape(-1, ref["crit"].shape[-1]), kpr, lens, spec.h_kv)
    B = spec.batch
    dref = oracle.draft(kv_h, qd, oidx.reshape(B, spec.h_kv, k_max), ocnt.reshape(B, spec.h_kv), scale)
    _gpu.assert_out(r["out"].cpu().numpy(), dref["out"], "oracle top-k draft")


def test_oracle_topk_draft_selecting_all_is_dense():
    """With K_b = L_b every token is selected, so the sparse draft equals the dense attention."""
    spec, w, kv_h, scale, kpr, k_max, r = _oracle_topk_case([700, 129, 1500], 22, select_all=True)
    assert r["cnt"].cpu().numpy().tolist() == np.repeat(kpr, spec.h_kv).tolist()
    _gpu.assert_out(r["out"].cpu().numpy(), r["dense"].cpu().numpy(), "select-all draft vs dense")
