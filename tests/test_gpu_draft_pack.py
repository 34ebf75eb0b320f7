"""Sparse draft attention through the row pack.  The writing call equals the plain draft bit for bit
(the same kernel, which also stores its tiles).  The reading calls are checked against the oracle
and against plain drafts of their own queries: bit-exact for fp32 caches (the plain chunked kernel
reading the pack); within 1e-4 relative for bf16 caches, whose reader runs one block per (request,
KV head) with a per-warp online softmax over the chunks instead of per-chunk partials merged by
log-sum-exp."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import (KVCache, SpecRound, binding, ssd_draft_attn, ssd_draft_attn_packed,
                                                 ssd_draft_pack_bytes, ssd_kv_append, ssd_status)
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_kv import _extended

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pack(kv, k_max, fill=None):
    n = ssd_draft_pack_bytes(kv, k_max)
    assert n > 0
    p = torch.empty(n + 256, dtype=torch.uint8, device=DEV)
    off = (-p.data_ptr()) % 256
    p = p[off:off + n]
    if fill is not None:
        p.fill_(fill)  # NaN bytes for bf16 / fp32 (0xff): rows the reader must not use
    return p


def _close(got, ref, what):
    """Reader against the plain draft: the same sums in another order (online rescaling)."""
    assert torch.allclose(got, ref, rtol=1e-4, atol=2e-5, equal_nan=False), \
        f"{what}: max |diff| {(got - ref).abs().max().item():.3g}"


def _lse_close(got, ref, what):
    fin = torch.isfinite(ref)
    assert torch.equal(fin, torch.isfinite(got)), what
    _close(got[fin], ref[fin], what)


def _queries(w, n):
    g = torch.Generator().manual_seed(99)
    q = torch.randn((n,) + tuple(w.q_draft[0].shape), generator=g)
    return q.to(w.q_draft.dtype).to(DEV)


CASES = [
    # (spec name, overrides, lens, k per request, k_max)
    ("qwen3_8b", dict(batch=3), [2049, 700, 64], [103, 35, 64], 128),
    ("qwen3_8b", dict(batch=2), [8192, 5000], [410, 250], 410),                 # 7 chunks: last-arriver merge
    ("qwen3_8b", dict(batch=2, h_q=40), [3000, 1200], [150, 0], 150),           # G = 5, one empty list
    ("qwen3_8b", dict(batch=2, h_q=128, h_kv=8), [600, 1000], [30, 300], 300),  # G = 16
    ("qwen3_8b", dict(batch=2, d=64, page_size=32), [1000, 333], [65, 17], 65),
    ("tiny", dict(), [512, 512], [64, 64], 64),                                 # fp32, d = 64
    ("tiny", dict(d=128, page_size=16, shuffled=True), [700, 129], [100, 7], 100),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{'_'.join(map(str, c[2]))}-k{c[4]}")
def test_pack_write_then_reads_equal_plain_drafts(case):
    _gpu.lib()
    name, over, lens, ks, k_max = case
    spec = W.scaled_spec(W.SPECS[name], name="dp", **over)
    w = W.make_workload(spec, seed=41 + k_max, device=DEV, lengths=lens)
    kv = KVCache.from_workload(w)
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), k_max, seed=k_max + 1)
    idx, cnt = idx.to(DEV), cnt.to(DEV)
    scale = _gpu.scale_of(spec)
    qs = _queries(w, 3)
    pack = _pack(kv, k_max, fill=0xFF)
    got = [ssd_draft_attn_packed(kv, qs[0], idx, cnt, scale, pack, binding.PACK_WRITE)]
    for j in (1, 2):
        got.append(ssd_draft_attn_packed(kv, qs[j], None, cnt, scale, pack, binding.PACK_READ, k_max=k_max))
    # The round's last read drops the pack from L2 afterwards: same results as a plain read.
    last = ssd_draft_attn_packed(kv, qs[2], None, cnt, scale, pack, binding.PACK_READ_DISCARD, k_max=k_max)
    ref = [ssd_draft_attn(kv, qs[j], idx, cnt, scale) for j in range(3)]
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(last["out"], got[2]["out"]) and torch.equal(last["lse"], got[2]["lse"])
    assert torch.equal(got[0]["out"], ref[0]["out"]) and torch.equal(got[0]["lse"], ref[0]["lse"])
    kv_h, reqs = _gpu.host_subset(w, None)
    for j in (1, 2):
        if spec.dtype != "bf16":
            assert torch.equal(got[j]["out"], ref[j]["out"]) and torch.equal(got[j]["lse"], ref[j]["lse"]), j
        else:
            _close(got[j]["out"], ref[j]["out"], f"read {j} out")
            _lse_close(got[j]["lse"], ref[j]["lse"], f"read {j} lse")
        o = oracle.draft(kv_h, qs[j].cpu()[reqs], idx.cpu()[reqs], cnt.cpu()[reqs], scale)
        _gpu.assert_out(got[j]["out"].cpu().numpy()[reqs], o["out"], f"read {j} out vs oracle")
        _gpu.assert_lse(got[j]["lse"].cpu().numpy()[reqs], o["lse"])


def test_pack_read_against_oracle_after_append():
    """Reading the pack after new tokens were appended past the old ends (the rows the pack holds are
    unchanged) still gives the oracle's draft over the selected tokens."""
    _gpu.lib()
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="dpa", batch=2)
    w = W.make_workload(spec, seed=7, device=DEV, lengths=[3000, 1500], spare_pages=4)
    kv = _extended(w, 3)
    k_max = 150
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor([150, 75], dtype=torch.int32), k_max, seed=8)
    scale = _gpu.scale_of(spec)
    pack = _pack(kv, k_max)
    qs = _queries(w, 2)
    ssd_draft_attn_packed(kv, qs[0], idx.to(DEV), cnt.to(DEV), scale, pack, binding.PACK_WRITE)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn((2, 3, spec.h_kv, spec.d), generator=g).to(kv.pool.dtype).to(DEV)
    v_new = torch.randn((2, 3, spec.h_kv, spec.d), generator=g).to(kv.pool.dtype).to(DEV)
    ssd_kv_append(kv, k_new, v_new)
    r = ssd_draft_attn_packed(kv, qs[1], None, cnt.to(DEV), scale, pack, binding.PACK_READ, k_max=k_max)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    kv_h, reqs = _gpu.host_subset(w, None)
    ref = oracle.draft(kv_h, qs[1].cpu()[reqs], idx[reqs], cnt[reqs], scale)
    _gpu.assert_out(r["out"].cpu().numpy()[reqs], ref["out"], "packed draft out")
    _gpu.assert_lse(r["lse"].cpu().numpy()[reqs], ref["lse"])


def test_pack_write_reports_index_faults_like_plain():
    _gpu.lib()
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="dpf", batch=2)
    w = W.make_workload(spec, seed=9, device=DEV, lengths=[1000, 800])
    kv = KVCache.from_workload(w)
    idx = torch.zeros((2, spec.h_kv, 64), dtype=torch.int32, device=DEV)
    idx[1, 3, 5] = 900  # past L = 800
    cnt = torch.full((2, spec.h_kv), 64, dtype=torch.int32, device=DEV)
    pack = _pack(kv, 64)
    scale = _gpu.scale_of(spec)
    a = ssd_draft_attn_packed(kv, w.q_draft[0], idx, cnt, scale, pack, binding.PACK_WRITE)
    torch.cuda.synchronize()
    assert ssd_status() == binding.FAULT_INDEX
    b = ssd_draft_attn(kv, w.q_draft[0], idx, cnt, scale)
    torch.cuda.synchronize()
    assert ssd_status() == binding.FAULT_INDEX
    assert torch.equal(a["out"], b["out"])
    # The faulting row was stored as zeros, so the reader matches the plain call and raises nothing.
    c = ssd_draft_attn_packed(kv, w.q_draft[0], None, cnt, scale, pack, binding.PACK_READ, k_max=64)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    _close(c["out"], a["out"], "read after faults")


def test_round_with_and_without_pack_full_size():
    """The full-size Qwen3-8B round: drafts through the row pack match plain drafts (the first bit for
    bit), and a replayed CUDA graph of the round reproduces the eager round exactly."""
    _gpu.lib()
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, device=DEV)
    k_max = int(w.k_per_req.max())
    scale = _gpu.scale_of(spec)
    a = SpecRound(KVCache.from_workload(w), spec.h_q, spec.n_cand, k_max, scale, pack_rows=False)
    b = SpecRound(KVCache.from_workload(w), spec.h_q, spec.n_cand, k_max, scale)
    oa = torch.empty((spec.k, spec.batch, spec.h_q, spec.d), dtype=torch.float32, device=DEV)
    ob = torch.empty_like(oa)
    a.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=oa)
    b.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=ob)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(oa[0], ob[0])
    _close(ob[1:], oa[1:], "drafts 2..k")
    eager = ob.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        ob.zero_()
        with torch.cuda.graph(g, stream=s):
            b.run(w.q_verify, w.q_draft, w.k_per_req, draft_outs=ob)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(eager, ob)
