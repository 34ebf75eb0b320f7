"""Block-granular path on the GPU: per-candidate block scores, block Top-K, union, block-sparse
attention over the union -- each stage against the oracle on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import (KVCache, ssd_block_sparse_attn, ssd_block_union, ssd_select_topk,
                                                 ssd_status, ssd_verify_attn)
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check_block_path(w, reqs=None):
    _gpu.lib()
    spec = w.spec
    scale = _gpu.scale_of(spec)
    kv = KVCache.from_workload(w)
    nb = (kv.max_seq_len + 63) // 64
    bs = torch.zeros((spec.batch, spec.h_kv, spec.n_cand, nb), device=DEV)
    ssd_verify_attn(kv, w.q_verify, spec.n_cand, scale, bscores=bs, want_scores=False)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    kv_h, reqs = _gpu.host_subset(w, reqs)
    ref = oracle.verify(kv_h, w.q_verify.cpu()[reqs], scale, per_candidate=True)
    bref = oracle.block_maxpool(ref["crit_cand"], kv_h.seq_lens, 64, nb)
    got = bs.cpu().numpy()[reqs]
    for i, L in enumerate(kv_h.seq_lens):
        n = (int(L) + 63) // 64
        e = bref[i, ..., :n]
        assert (np.abs(got[i, ..., :n] - e) <= _gpu.SCORE_RTOL * np.abs(e) + _gpu.SCORE_ATOL).all()
    # Block Top-K and union on the oracle's fp32 block scores, both sides.
    B = len(reqs)
    S = np.zeros((B, spec.h_kv, spec.n_cand, nb), np.float32)
    for i, L in enumerate(kv_h.seq_lens):
        n = (int(L) + 63) // 64
        S[i, ..., :n] = bref[i, ..., :n]
    kb = spec.top_blocks
    lens = torch.as_tensor(kv_h.seq_lens)
    ks = torch.full((B,), kb, dtype=torch.int32)
    gi, gc = ssd_select_topk(torch.from_numpy(S).to(DEV), lens.to(DEV), ks.to(DEV), kb, spec.h_kv * spec.n_cand,
                             len_div=64, max_len=nb)
    oi, oc = oracle.topk(S.reshape(-1, nb), lens.numpy(), ks.numpy(), kb, spec.h_kv * spec.n_cand, 64)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gi.cpu().numpy(), oi)
    np.testing.assert_array_equal(gc.cpu().numpy(), oc)
    blocks = oi.reshape(B * spec.h_kv, spec.n_cand, kb)
    bcnt = oc.reshape(B * spec.h_kv, spec.n_cand)
    ui, um, uc = ssd_block_union(torch.from_numpy(blocks).to(DEV), torch.from_numpy(bcnt).to(DEV), nb)
    oui, oum, ouc = oracle.block_union(blocks, bcnt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(uc.cpu().numpy(), ouc)
    np.testing.assert_array_equal(ui.cpu().numpy(), oui)
    np.testing.assert_array_equal(um.cpu().numpy().view(np.uint32), oum)
    # Block-sparse attention over the union, on the oracle's union, for the sampled requests.
    full_ui = torch.full((spec.batch * spec.h_kv, oui.shape[1]), -1, dtype=torch.int32)
    full_um = torch.zeros((spec.batch * spec.h_kv, oui.shape[1]), dtype=torch.int32)
    full_uc = torch.zeros((spec.batch * spec.h_kv,), dtype=torch.int32)
    for i, b in enumerate(reqs):
        full_ui[b * spec.h_kv:(b + 1) * spec.h_kv] = torch.from_numpy(oui[i * spec.h_kv:(i + 1) * spec.h_kv])
        full_um[b * spec.h_kv:(b + 1) * spec.h_kv] = torch.from_numpy(oum[i * spec.h_kv:(i + 1) * spec.h_kv].view(np.int32))
        full_uc[b * spec.h_kv:(b + 1) * spec.h_kv] = torch.from_numpy(ouc[i * spec.h_kv:(i + 1) * spec.h_kv])
    r = ssd_block_sparse_attn(kv, w.q_verify, spec.n_cand, full_ui.to(DEV), full_um.to(DEV), full_uc.to(DEV), scale)
    aref = oracle.block_attn(kv_h, w.q_verify.cpu()[reqs], blocks.reshape(B, spec.h_kv, spec.n_cand, kb),
                             bcnt.reshape(B, spec.h_kv, spec.n_cand), 64, scale)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    _gpu.assert_out(r["out"].cpu().numpy()[reqs], aref["out"], "block-sparse out")
    _gpu.assert_lse(r["lse"].cpu().numpy()[reqs], aref["lse"])


def test_block_path_small():
    spec = W.scaled_spec(W.SPECS["block_131k"], name="blk", batch=3)
    _check_block_path(W.make_workload(spec, seed=13, device=DEV, lengths=[8192 + 33, 3000, 1100]))


def test_block_path_full_size_sampled():
    w = W.make_workload(W.SPECS["block_131k"], device=DEV)
    _check_block_path(w, reqs=[0, 7])


# Pages of 8 and 32 tokens (a union block's rows in 8 or 2 runs of the pool), R = 40 (four row tiles:
# the block-sparse kernel without its shared row table), and d = 64.
@pytest.mark.parametrize("over,lens", [
    (dict(batch=2, page_size=8), [5000, 2100]),
    (dict(batch=2, page_size=32), [6000, 777]),
    (dict(batch=2, h_q=64), [4100, 2500]),
    (dict(batch=2, d=64), [3000, 1500]),
], ids=["ps8", "ps32", "R40", "d64"])
def test_block_path_shapes(over, lens):
    spec = W.scaled_spec(W.SPECS["block_131k"], name="blks", **over)
    _check_block_path(W.make_workload(spec, seed=21, device=DEV, lengths=lens))
