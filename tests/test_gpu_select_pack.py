"""ssd_verify_select_packed: the fused verify-select that also stores the selected K and V rows in the
draft's row pack.  Its pack is, byte for byte, the pack an SSD_PACK_WRITE draft over the same
selection stores (both buffers start from the same fill pattern); its other outputs equal
ssd_verify_select's; drafts reading it equal the plain drafts on that selection (bit for bit on the
fp32 path, which reads the pack through the chunk kernel) and the oracle drafts."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import KVCache, binding, ssd_draft_attn, ssd_status, ssd_verify_select
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _pack_buffer(n: int, fill: int) -> torch.Tensor:
    buf = torch.full((n + 256,), fill, dtype=torch.uint8, device=DEV)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + n]


def _check(w, ks=None, k_max=None, n_drafts=2, reqs=None):
    _gpu.lib()
    spec = w.spec
    kv = KVCache.from_workload(w)
    scale = _gpu.scale_of(spec)
    ks = w.k_per_req if ks is None else ks
    k_max = int(ks.max()) if k_max is None else k_max
    nbytes = binding.ssd_draft_pack_bytes(kv, k_max)
    p_sel = _pack_buffer(nbytes, 0xA5)
    f = ssd_verify_select(kv, w.q_verify, spec.n_cand, scale, ks, k_max, pack=p_sel)
    g = ssd_verify_select(kv, w.q_verify, spec.n_cand, scale, ks, k_max)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    for name in ("out", "lse", "scores", "idx", "cnt"):
        assert torch.equal(f[name], g[name]), name
    B, hkv = kv.batch, kv.h_kv
    idx = f["idx"].view(B, hkv, k_max)
    cnt = f["cnt"].view(B, hkv)
    p_draft = _pack_buffer(nbytes, 0xA5)
    binding.ssd_draft_attn_packed(kv, w.q_draft[0], idx, cnt, scale, p_draft, binding.PACK_WRITE)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert torch.equal(p_sel, p_draft), "pack stored by the selection differs from the first draft's"
    fp32 = spec.dtype != "bf16"
    kv_h, sub = _gpu.host_subset(w, reqs)
    for j in range(min(n_drafts, spec.k)):
        r = binding.ssd_draft_attn_packed(kv, w.q_draft[j], idx, cnt, scale, p_sel, binding.PACK_READ)
        d = ssd_draft_attn(kv, w.q_draft[j], idx, cnt, scale)
        torch.cuda.synchronize()
        assert ssd_status() == 0
        if fp32:
            assert torch.equal(r["out"], d["out"])
        else:
            torch.testing.assert_close(r["out"], d["out"], rtol=1e-4, atol=1e-5)
        oidx = idx.cpu().numpy()[sub]
        ocnt = cnt.cpu().numpy()[sub]
        dref = oracle.draft(kv_h, w.q_draft[j].cpu()[sub], oidx, ocnt, scale)
        _gpu.assert_out(r["out"].cpu().numpy()[sub], dref["out"], f"packed draft {j}")
    return f


CASES = [
    # (lens, h_q, h_kv, d, n_cand, page_size)
    ([700, 129, 5000], 32, 8, 128, 5, 16),   # one to 250 selected rows (four chunks), ragged
    ([4097, 2048], 32, 8, 128, 7, 16),
    ([1111, 2222], 8, 2, 64, 3, 64),         # d = 64, pages of 64
    ([5], 4, 2, 128, 5, 16),                 # L = n_cand: one selected row
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{'_'.join(map(str, c[0]))}-d{c[3]}-ps{c[5]}")
def test_select_pack_equals_first_draft_pack(case):
    lens, h_q, h_kv, d, nc, ps = case
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="spack", batch=len(lens), h_q=h_q, h_kv=h_kv, d=d, k=nc - 1,
                         page_size=ps)
    w = W.make_workload(spec, seed=61 + sum(lens), device=DEV, lengths=lens, spare_pages=3)
    _check(w)


def test_select_pack_fp32_and_select_all():
    """fp32 cache (pack read through the chunk kernel, bit for bit); K = L packs every token."""
    w = W.make_workload(W.SPECS["tiny"], device=DEV)
    _check(w)
    _check(w, ks=w.seq_lens.clone())


def test_select_pack_long_rows_finalize_path():
    """Rows longer than the criticality pass keeps in shared memory: the finalize's last token block
    selects, and packs, the row."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="spack_long", batch=2)
    w = W.make_workload(spec, seed=71, device=DEV, lengths=[45000, 3000])
    assert w.seq_lens.max().item() > 40960
    _check(w, n_drafts=1)


def test_select_pack_full_size_round():
    """The Qwen3-8B round as the benchmark runs it: the pack written by the verify-select and read by
    all four drafts, on sampled requests against the oracle drafts."""
    w = W.make_workload(W.SPECS["qwen3_8b"], device=DEV)
    _check(w, n_drafts=4, reqs=[2, 19, 30])
