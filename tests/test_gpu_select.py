"""Top-K selection and block union on the GPU: bit-exact against the oracle on the same fp32
score tensors (generator-made rows with many exact ties, and the oracle's own criticality)."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import ssd_block_union, ssd_select_topk, ssd_status
from sparse_self_speculative_verify_gb300 import binding
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _both(scores, lens, ks, k_max, rows_per_group=1, len_div=1, max_len=None, expect_status=0):
    _gpu.lib()
    s = torch.as_tensor(scores).contiguous()
    lens_t = torch.as_tensor(np.asarray(lens, np.int32))
    ks_t = torch.as_tensor(np.asarray(ks, np.int32))
    gi, gc = ssd_select_topk(s.to(DEV), lens_t.to(DEV), ks_t.to(DEV), k_max, rows_per_group, len_div, max_len)
    torch.cuda.synchronize()
    assert ssd_status() == expect_status
    oi, oc = oracle.topk(s.reshape(-1, s.shape[-1]).numpy(), lens_t.numpy(),
                         np.minimum(ks_t.numpy(), k_max) if expect_status else ks_t.numpy(), k_max,
                         rows_per_group, len_div)
    np.testing.assert_array_equal(gc.cpu().numpy(), oc)
    np.testing.assert_array_equal(gi.cpu().numpy(), oi)


@pytest.mark.parametrize("length,k", [(1, 1), (7, 3), (100, 5), (2049, 103), (5000, 250), (8192, 410), (32768, 1639)])
def test_topk_tie_heavy(length, k):
    rows = 6
    s = W.random_scores(rows, length, seed=length + k, ties=True)
    _both(s, [length] * rows, [k] * rows, k)


def test_topk_distinct_values():
    s = W.random_scores(16, 4000, seed=1, ties=False)
    _both(s, [4000, 3999, 2500, 17] * 4, [200, 200, 125, 1] * 4, 200)


def test_topk_ragged_groups():
    """rows_per_group > 1, per-group lengths shorter than the stride, K = L, K = 0."""
    s = W.random_scores(4 * 8, 1000, seed=3)
    _both(s, [1000, 999, 64, 0], [50, 999, 64, 0], 999, rows_per_group=8)


def test_topk_constant_and_zero_rows():
    s = torch.zeros((3, 300))
    s[1] = 0.25
    s[2, 150:] = -0.0  # ranks equal to +0.0
    _both(s, [300] * 3, [10, 10, 160], 160)


def test_topk_long_rows_global_path():
    """Rows longer than the shared-memory staging limit are read from global memory each pass."""
    s = W.random_scores(2, 131072, seed=5)
    _both(s, [131072, 100000], [6554, 5000], 6554)


def test_topk_k_over_kmax_faults_and_truncates():
    s = W.random_scores(2, 500, seed=6)
    _both(s, [500, 500], [40, 40], 20, expect_status=binding.FAULT_KMAX)


def test_topk_on_oracle_scores():
    """The oracle's own criticality (cast to fp32) selected by both sides."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="sel", batch=3)
    w = W.make_workload(spec, seed=4, device="cpu", lengths=[3000, 2049, 640])
    kv = oracle.PagedKV(w.pool, w.page_table, w.seq_lens)
    ref = oracle.verify(kv, w.q_verify, _gpu.scale_of(spec))
    S = torch.from_numpy(ref["crit"].astype(np.float32))
    kmax = int(w.k_per_req.max())
    _both(S.view(-1, S.shape[-1]), w.seq_lens.numpy(), w.k_per_req.numpy(), kmax, rows_per_group=spec.h_kv)


def test_block_topk_len_div():
    """Block selection: rows of n_cand candidates per KV head, lengths ceil(L / 64)."""
    L = [131072, 70000]
    nb = (max(L) + 63) // 64
    s = W.random_scores(2 * 8 * 5, nb, seed=8)
    _both(s, L, [16, 16], 16, rows_per_group=8 * 5, len_div=64, max_len=nb)


def test_block_union_matches_oracle():
    _gpu.lib()
    gen = torch.Generator().manual_seed(12)
    U, nc, kb, nblk = 37, 5, 16, 2048
    blocks = torch.stack([torch.stack([torch.randperm(nblk if u % 3 else 40, generator=gen)[:kb] for _ in range(nc)])
                          for u in range(U)]).to(torch.int32)
    bcnt = torch.randint(0, kb + 1, (U, nc), generator=gen).to(torch.int32)
    bcnt[0] = kb
    gi, gm, gc = ssd_block_union(blocks.to(DEV), bcnt.to(DEV), nblk)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    oi, om, oc = oracle.block_union(blocks.numpy(), bcnt.numpy())
    np.testing.assert_array_equal(gc.cpu().numpy(), oc)
    np.testing.assert_array_equal(gi.cpu().numpy(), oi)
    np.testing.assert_array_equal(gm.cpu().numpy().view(np.uint32), om)


def test_topk_threshold_bin_paths():
    """Rows built for each way the shared-memory selection narrows its threshold bin (the bin of the
    keys' top 12 bits that holds the K-th largest): more than 1024 keys in the bin (three passes over
    the row); more than 32 keys left after the bin's next 8 bits (two more passes over the gathered
    keys); and a few left (their ranks across a warp)."""
    n = 5000
    rng = np.random.default_rng(31)
    rows = np.zeros((3, n), np.float32)
    # 3000 distinct values in [1, 1.1) (one 12-bit bin: sign, exponent and 3 mantissa bits), 2000 in [2, 4).
    rows[0, :3000] = 1.0 + rng.permutation(3000).astype(np.float32) * np.float32(2.0 ** -15)
    rows[0, 3000:] = rng.uniform(2.0, 4.0, 2000).astype(np.float32)
    # 400 values in the bin: 120 of them share their top 20 bits (differ in the low 12 only).
    rows[1, :280] = 1.0 + (4096 + rng.permutation(280)).astype(np.float32) * np.float32(2.0 ** -19)
    rows[1, 280:400] = 1.0 + rng.permutation(120).astype(np.float32) * np.float32(2.0 ** -23)
    rows[1, 400:] = rng.uniform(0.0, 0.5, n - 400).astype(np.float32)
    rows[2] = rng.uniform(0.0, 1.0, n).astype(np.float32)
    for r in range(3):
        rng.shuffle(rows[r])
    # Row 0: K inside the 3000-key bin; row 1: inside the 120 shared keys (280 lie above them); row 2: 5 %.
    _both(torch.from_numpy(rows), [n] * 3, [2500, 340, 250], 2500)
