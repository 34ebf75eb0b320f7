"""Unified verify/draft launch on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import KVCache, ssd_status, ssd_unified_attn
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_and_check(w, reqs=None):
    _gpu.lib()
    spec = w.spec
    k_max = int(w.k_per_req.max())
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, w.k_per_req, k_max, seed=w.seed)
    kv = KVCache.from_workload(w)
    scale = _gpu.scale_of(spec)
    r = ssd_unified_attn(kv, w.phase, w.q_verify, w.q_draft[0], spec.n_cand, idx.to(DEV), cnt.to(DEV), scale)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    phase = w.phase.cpu().numpy()
    reqs = list(range(spec.batch)) if reqs is None else reqs
    vreq = [b for b in reqs if phase[b] == 1]
    dreq = [b for b in reqs if phase[b] == 0]
    assert vreq and dreq
    kv_h, vreq = _gpu.host_subset(w, vreq)
    ref = oracle.verify(kv_h, w.q_verify.cpu()[vreq], scale)
    _gpu.assert_out(r["out_verify"].cpu().numpy()[vreq], ref["out"], "unified verify out")
    _gpu.assert_lse(r["lse_verify"].cpu().numpy()[vreq], ref["lse"])
    _gpu.assert_scores(r["scores"].cpu().numpy()[vreq], ref["crit"], kv_h.seq_lens)
    kv_d, dreq = _gpu.host_subset(w, dreq)
    dref = oracle.draft(kv_d, w.q_draft[0].cpu()[dreq], idx[dreq], cnt[dreq], scale)
    _gpu.assert_out(r["out_draft"].cpu().numpy()[dreq], dref["out"], "unified draft out")
    _gpu.assert_lse(r["lse_draft"].cpu().numpy()[dreq], dref["lse"])


def test_unified_small():
    spec = W.scaled_spec(W.SPECS["qwen3_14b_unified"], name="uni", batch=10, len_lo=600, len_hi=4096,
                         len_median=2000.0, verify_prob=0.4)
    _run_and_check(W.make_workload(spec, seed=5, device=DEV))


def test_unified_persistent_launch_d64():
    """d = 64 (no tcgen05 verify): one persistent launch mixes the verify and draft items."""
    spec = W.scaled_spec(W.SPECS["qwen3_14b_unified"], name="uni64", batch=9, d=64, len_lo=600, len_hi=3000,
                         len_median=1500.0, verify_prob=0.4)
    _run_and_check(W.make_workload(spec, seed=6, device=DEV))


def test_unified_full_size_sampled():
    spec = W.SPECS["qwen3_14b_unified"]
    w = W.make_workload(spec, device=DEV)
    phase = w.phase.cpu().numpy()
    v = [b for b in range(spec.batch) if phase[b]][:2]
    d = [b for b in range(spec.batch) if not phase[b]][:3]
    _run_and_check(w, reqs=v + d)
