"""Verify attention + criticality on the GPU against the float64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import KVCache, ssd_status, ssd_verify_attn
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(w, scores=True, bscores=False):
    _gpu.lib()
    kv = KVCache.from_workload(w)
    bs = None
    if bscores:
        nb = (kv.max_seq_len + 63) // 64
        bs = torch.full((w.spec.batch, w.spec.h_kv, w.spec.n_cand, nb), -1.0, device=DEV)
    r = ssd_verify_attn(kv, w.q_verify, w.spec.n_cand, _gpu.scale_of(w.spec), bscores=bs, want_scores=scores)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    return r


def _compare(w, r, reqs=None, block=False):
    kv_h, reqs = _gpu.host_subset(w, reqs)
    ref = oracle.verify(kv_h, w.q_verify.cpu()[reqs], _gpu.scale_of(w.spec), per_candidate=block)
    _gpu.assert_out(r["out"].cpu().numpy()[reqs], ref["out"], "verify out")
    _gpu.assert_lse(r["lse"].cpu().numpy()[reqs], ref["lse"])
    lens = kv_h.seq_lens
    if r["scores"] is not None:
        _gpu.assert_scores(r["scores"].cpu().numpy()[reqs], ref["crit"], lens)
    if block:
        bref = oracle.block_maxpool(ref["crit_cand"], lens, 64)
        got = r["bscores"].cpu().numpy()[reqs]
        for i, L in enumerate(lens):
            nb = (int(L) + 63) // 64
            g = got[i, :, :, :nb].astype(np.float64)
            e = bref[i, :, :, :nb]
            assert (np.abs(g - e) <= _gpu.SCORE_RTOL * np.abs(e) + _gpu.SCORE_ATOL).all(), "block scores"
    return ref


def test_verify_tiny_fp32():
    """The 2 x 512, 8/2-head, d=64, fp32, contiguous workload: every output."""
    w = W.make_workload(W.SPECS["tiny"], device=DEV)
    _compare(w, _run(w))


SMALL = [
    # (B, lens, h_q, h_kv, d, n_cand, page_size)
    (3, [700, 129, 1025], 32, 8, 128, 5, 16),   # R = 20, several splits and ragged tails
    (2, [513, 64], 8, 8, 64, 1, 16),            # G = 1, n_cand = 1, d = 64
    (2, [1000, 77], 40, 8, 128, 5, 8),          # R = 25 (Qwen3-14B grouping), page 8
    (2, [600, 300], 16, 1, 128, 4, 32),         # G = 16, R = 64 (four row tiles)
    (1, [5], 4, 2, 128, 5, 16),                 # L = n_cand: the first candidate sees one token
    (2, [2048, 1536], 32, 8, 128, 7, 16),       # R = 28 (k = 6)
    (2, [1111, 2222], 8, 2, 64, 3, 64),         # d = 64, R = 12, page 64
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}-L{'_'.join(map(str, c[1]))}-G{c[2]//c[3]}-d{c[4]}-nc{c[5]}-ps{c[6]}")
def test_verify_small_bf16(case):
    B, lens, h_q, h_kv, d, nc, ps = case
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="small", batch=B, h_q=h_q, h_kv=h_kv, d=d, k=nc - 1,
                         page_size=ps)
    w = W.make_workload(spec, seed=11 + sum(lens), device=DEV, lengths=lens, spare_pages=5)
    _compare(w, _run(w))


def test_verify_fp32_d128():
    spec = W.scaled_spec(W.SPECS["tiny"], name="f32", batch=2, d=128, page_size=16, shuffled=True)
    w = W.make_workload(spec, seed=5, device=DEV, lengths=[600, 97])
    _compare(w, _run(w))


def test_verify_block_scores():
    spec = W.scaled_spec(W.SPECS["block_131k"], name="blk", batch=2)
    w = W.make_workload(spec, seed=3, device=DEV, lengths=[4096 + 17, 1000])
    _compare(w, _run(w, bscores=True), block=True)


def test_verify_without_scores():
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="nosc", batch=2)
    w = W.make_workload(spec, seed=9, device=DEV, lengths=[900, 333])
    r = _run(w, scores=False)
    assert r["scores"] is None
    _compare(w, r)


def test_verify_paging_invariance():
    """Identity and shuffled page tables give bit-identical GPU results."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="pg", batch=3)
    lens = [1500, 800, 2049]
    a = W.make_workload(spec, seed=21, device=DEV, lengths=lens)
    b = W.make_workload(W.scaled_spec(spec, shuffled=False), seed=21, device=DEV, lengths=lens)
    assert torch.equal(a.q_verify, b.q_verify)
    ra, rb = _run(a), _run(b)
    for k in ("out", "lse", "scores"):
        assert torch.equal(ra[k], rb[k]), k


@pytest.mark.parametrize("name", ["qwen3_8b", "b128_l8k"])
def test_verify_full_size_sampled(name):
    """The full-size workload in the benchmark's launch configuration; the oracle recomputes a
    sample of requests (every head, every candidate and every token of them)."""
    spec = W.SPECS[name]
    w = W.make_workload(spec, device=DEV)
    r = _run(w)
    B = spec.batch
    _compare(w, r, reqs=[0, B // 3, B - 1])


def test_verify_many_short_requests():
    """300 ragged requests of 5 to 700 tokens (some a single tile, some one split of several): the
    verify's item decode searches the per-request item prefix in more than one round.  Every request
    against the oracle."""
    rng = np.random.default_rng(17)
    lens = [int(x) for x in rng.integers(5, 701, 300)]
    lens[:4] = [5, 128, 129, 700]
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="many", batch=len(lens))
    w = W.make_workload(spec, seed=23, device=DEV, lengths=lens)
    _compare(w, _run(w))
