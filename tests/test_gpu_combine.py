"""ssd_combine, the split-KV combine (log-sum-exp merge) exported by the C ABI, against the oracle.

SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
Sparse Attention") §4.1: the verify caches each part's log-sum-exp, so attention over disjoint parts
of the token set merges into attention over their union.  The split partials here are made by the
oracle (drafts over disjoint index subsets of a seeded workload, and seeded random partials), never
by the GPU; the GPU merge is compared with the oracle merge and with the oracle draft over the union.
"""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import ssd_combine, ssd_status
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu_combine(o_parts, lse_parts):
    _gpu.lib()
    o = torch.from_numpy(np.ascontiguousarray(o_parts, np.float32)).to(DEV)
    lp = torch.from_numpy(np.ascontiguousarray(lse_parts, np.float32)).to(DEV)
    out, lse = ssd_combine(o, lp)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("d", [64, 128])
def test_combine_of_split_drafts_equals_union_draft(d):
    """Drafts over S disjoint index subsets (some empty), merged on the GPU, against the oracle's
    merge of the same partials and the oracle draft over the union."""
    name = "qwen3_8b" if d == 128 else "tiny"
    spec = W.scaled_spec(W.SPECS[name], name="comb", batch=3, dtype="bf16", page_size=16)
    lens = [3000, 777, 64]
    w = W.make_workload(spec, seed=40 + d, device="cpu", lengths=lens)
    kv_h, _ = _gpu.host_subset(w)
    scale = _gpu.scale_of(spec)
    k_max = 300
    ks = torch.tensor([300, 120, 33], dtype=torch.int32)
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, ks, k_max, seed=5)
    idx, cnt = idx.numpy(), cnt.numpy()
    q = w.q_draft[0]
    whole = oracle.draft(kv_h, q, idx, cnt, scale)
    # Split every list at fixed fractions into 5 parts; part 1 is always empty.
    fracs = [0.0, 0.3, 0.3, 0.55, 0.9, 1.0]
    parts_o, parts_l = [], []
    for s in range(5):
        pidx = np.full_like(idx, -1)
        pcnt = np.zeros_like(cnt)
        for b in range(spec.batch):
            for g in range(spec.h_kv):
                n = int(cnt[b, g])
                lo, hi = int(fracs[s] * n), int(fracs[s + 1] * n)
                pidx[b, g, :hi - lo] = idx[b, g, lo:hi]
                pcnt[b, g] = hi - lo
        r = oracle.draft(kv_h, q, pidx, pcnt, scale)
        parts_o.append(r["out"].reshape(-1, d))
        parts_l.append(r["lse"].reshape(-1))
    o_parts = np.stack(parts_o, axis=1).astype(np.float32)   # [B*h_q, 5, d]
    l_parts = np.stack(parts_l, axis=1).astype(np.float32)   # [B*h_q, 5]
    assert np.isneginf(l_parts[:, 1]).all()
    out, lse = _gpu_combine(o_parts, l_parts)
    ref_out, ref_lse = oracle.combine(o_parts, l_parts)
    _gpu.assert_out(out, ref_out, "combine vs oracle combine", tol=1e-5)
    _gpu.assert_lse(lse, ref_lse, "combine lse vs oracle combine")
    _gpu.assert_out(out, whole["out"].reshape(-1, d), "combine vs union draft")
    _gpu.assert_lse(lse, whole["lse"].reshape(-1), "combine lse vs union draft")


@pytest.mark.parametrize("n_splits,d", [(1, 128), (3, 64), (7, 128), (40, 128), (2, 40), (0, 128)])
def test_combine_random_partials(n_splits, d):
    """Seeded random partials with empty splits (-inf), one all-empty row and widely spread LSEs,
    against the oracle merge; one split is the identity bit for bit; no split gives 0 and -inf."""
    rng = np.random.default_rng(100 + n_splits * 7 + d)
    rows = 37
    o = rng.standard_normal((rows, n_splits, d)).astype(np.float32)
    l = (rng.standard_normal((rows, n_splits)) * 6.0).astype(np.float32)
    if n_splits:
        l[rng.random((rows, n_splits)) < 0.25] = -np.inf
        l[5, :] = -np.inf                       # all-empty row
        l[6, :] = 80.0                          # large equal LSEs
    out, lse = _gpu_combine(o, l)
    ref_out, ref_lse = oracle.combine(o, l)
    _gpu.assert_out(out, ref_out, "combine out", tol=1e-5)
    _gpu.assert_lse(lse, ref_lse, "combine lse")
    if n_splits == 0:
        assert np.isneginf(lse).all() and not out.any()
    else:
        assert np.isneginf(lse[5]) and not out[5].any()
    if n_splits == 1:
        fin = np.isfinite(l[:, 0])
        np.testing.assert_array_equal(out[fin], o[fin, 0])
        np.testing.assert_array_equal(lse[fin], l[fin, 0])
