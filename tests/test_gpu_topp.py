"""Top-p selection on the GPU against the oracle.

The per-row count K must equal the oracle's (sorted prefix sums in fp64) except where the
cumulative sum lies within the kernel's stated fixed-point resolution of the target; there both
counts must reach the target within that bound.  Given the count, the kept indices are the Top-K
set and are compared bit-exactly with the oracle's Top-K at the GPU's count."""

import math

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import binding, ssd_select_topp, ssd_status
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _resolution(row: np.ndarray) -> float:
    """Absolute bound on the kernel's fixed-point rounding over a whole row: n units of
    2^(ceil(log2 n) - 62) times the power of two just above the row maximum."""
    n = row.size
    if n == 0:
        return 0.0
    lg = max(n - 1, 0).bit_length()
    vmax = float(row.max())
    if vmax <= 0.0:
        return 0.0
    e = max(int(np.float32(vmax).view(np.uint32) >> 23) & 255, 1)
    return n * math.ldexp(1.0, lg - 62 + e - 126)


def _count_ok(row: np.ndarray, p: float, k: int, k_max: int) -> bool:
    """k is min(K, k_max) for a K whose prefix reaches p * total within the row's resolution and
    whose prefix one shorter does not."""
    s = np.sort(row.astype(np.float64))[::-1]
    pre = np.concatenate([[0.0], np.cumsum(s)])
    target = p * pre[-1]
    tol = _resolution(row) + abs(target) * 2.0 ** -50
    reach = pre >= target - tol
    short = np.concatenate([[True], pre[:-1] < target + tol])
    K = np.nonzero(reach & short)[0]
    return bool((np.minimum(K, k_max) == k).any())


def _both(scores, lens, p, k_max, rows_per_group=1, len_div=1, max_len=None, expect_status=0, exact_rows=None):
    _gpu.lib()
    s = torch.as_tensor(scores, dtype=torch.float32).contiguous()
    s2 = s.reshape(-1, s.shape[-1])
    lens_n = np.asarray(lens, np.int32)
    p32 = float(np.float32(p))
    gi, gc, gk = ssd_select_topp(s.to(DEV), torch.from_numpy(lens_n).to(DEV), p32, k_max, rows_per_group,
                                 len_div, max_len)
    torch.cuda.synchronize()
    assert ssd_status() == expect_status
    gk, gc, gi = gk.cpu().numpy(), gc.cpu().numpy(), gi.cpu().numpy()
    np.testing.assert_array_equal(gc, gk)
    if expect_status:
        return gi, gc, gk
    _, _, ok_k = oracle.topp(s2.numpy(), lens_n, p32, k_max, rows_per_group, len_div)
    row_len = np.repeat((lens_n + len_div - 1) // len_div, rows_per_group)
    differ = np.nonzero(ok_k != gk)[0]
    for r in differ:
        assert _count_ok(s2[r, :row_len[r]].numpy(), p32, int(gk[r]), k_max), (r, int(gk[r]), int(ok_k[r]))
    if exact_rows is not None:
        assert differ.size == 0 or not exact_rows, differ
    oi, oc = oracle.topk(s2.numpy(), np.repeat(lens_n, rows_per_group), gk, k_max, 1, len_div)
    np.testing.assert_array_equal(gc, oc)
    np.testing.assert_array_equal(gi, oi)
    return gi, gc, gk


@pytest.mark.parametrize("length", [1, 7, 513, 2049, 5000, 8192, 40960])
@pytest.mark.parametrize("p", [0.5, 0.9, 0.99, 1.0])
def test_topp_random_rows(length, p):
    s = W.random_scores(6, length, seed=length + int(p * 100), ties=False)
    _both(s, [length] * 6, p, length)


@pytest.mark.parametrize("length", [100, 4097, 32768])
def test_topp_tie_heavy_rows(length):
    """Many exactly equal values (eighths) and zeros: the count lands inside runs of ties."""
    s = W.random_scores(8, length, seed=3 * length, ties=True)
    for p in (0.25, 0.5, 0.75, 0.95, 1.0):
        _both(s, [length] * 8, p, length)


def test_topp_equal_values_closed_form():
    """A row of n equal values keeps ceil(p * n) of them (the lowest indices)."""
    n = 1000
    s = torch.full((4, n), 0.125)
    for p in (0.001, 0.3, 0.5, 0.999, 1.0):
        gi, gc, _ = _both(s, [n, 999, 500, 1], p, n, exact_rows=True)
        want = [math.ceil(float(np.float32(p)) * m) for m in (n, 999, 500, 1)]
        assert gc.tolist() == want
        assert gi[0, :want[0]].tolist() == list(range(want[0]))


def test_topp_cap_zero_p_and_empty_rows():
    s = W.random_scores(4 * 8, 3000, seed=9, ties=False)
    _, gc, _ = _both(s, [3000, 2999, 1, 0], 0.95, 64, rows_per_group=8)
    assert (gc[:16] == 64).all() and (gc[16:24] == 1).all() and (gc[24:] == 0).all()
    _, gc, _ = _both(s, [3000, 2999, 1, 0], 0.0, 64, rows_per_group=8, exact_rows=True)
    assert (gc == 0).all()


def test_topp_zero_rows_and_signed_zero():
    s = torch.zeros((3, 300))
    s[1, 17] = 1.0
    s[2, 150:] = -0.0
    _, gc, _ = _both(s, [300] * 3, 0.9, 300, exact_rows=True)
    assert gc.tolist() == [0, 1, 0]


def test_topp_skewed_row_one_dominant():
    """One entry holding most of the mass: p below its share keeps exactly that entry."""
    s = W.random_scores(2, 6000, seed=11, ties=False) * 1e-4
    s[0, 4321] = 10.0
    s[1, 0] = 10.0
    _, gc, _ = _both(s, [6000, 6000], 0.9, 6000)
    assert gc.tolist() == [1, 1]


def test_topp_long_rows_global_path():
    """Rows longer than the shared-memory staging limit are read from global memory each pass."""
    s = W.random_scores(2, 131072, seed=5, ties=False)
    _both(s, [131072, 100000], 0.9, 131072)


def test_topp_block_rows_len_div():
    L = [131072, 70000]
    nb = (max(L) + 63) // 64
    s = W.random_scores(2 * 8 * 5, nb, seed=8)
    _both(s, L, 0.8, nb, rows_per_group=8 * 5, len_div=64, max_len=nb)


def test_topp_on_oracle_scores():
    """The oracle's own criticality (cast to fp32): the distribution the draft selects from."""
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="topp", batch=3)
    w = W.make_workload(spec, seed=4, device="cpu", lengths=[3000, 2049, 640])
    kv = oracle.PagedKV(w.pool, w.page_table, w.seq_lens)
    ref = oracle.verify(kv, w.q_verify, _gpu.scale_of(spec))
    S = torch.from_numpy(ref["crit"].astype(np.float32))
    for p in (0.5, 0.9, 0.99):
        _both(S.view(-1, S.shape[-1]), w.seq_lens.numpy(), p, 2048, rows_per_group=spec.h_kv)


def test_topp_negative_or_nan_rows_fault():
    s = W.random_scores(3, 500, seed=13, ties=False)
    s[0, 7] = -0.5
    s[2, 400] = float("nan")
    gi, gc, gk = _both(s, [500] * 3, 0.9, 500, expect_status=binding.FAULT_VALUE)
    assert gk[0] == 0 and gk[2] == 0 and gk[1] > 0
    assert (gi[0] == -1).all() and (gi[2] == -1).all()


def test_topp_argument_errors():
    _gpu.lib()
    s = torch.zeros((2, 10), device=DEV)
    lens = torch.tensor([10, 10], dtype=torch.int32, device=DEV)
    for bad_p in (-0.1, 1.5, float("nan")):
        with pytest.raises(binding.SSDError):
            ssd_select_topp(s, lens, bad_p, 4, 1)
    with pytest.raises(binding.SSDError):
        ssd_select_topp(s, lens, 0.5, 4, 1, max_len=11)


def test_topp_full_size_on_verify_scores():
    """The full-size Qwen3-8B verify's criticality rows (32 requests x 8 KV heads, up to 8192 tokens),
    selected at p = 0.9 in the launch the round would use; sampled rows against the oracle."""
    _gpu.lib()
    from sparse_self_speculative_verify_gb300 import KVCache, ssd_verify_attn
    spec = W.SPECS["qwen3_8b"]
    w = W.make_workload(spec, device=DEV)
    kv = KVCache.from_workload(w)
    r = ssd_verify_attn(kv, w.q_verify, spec.n_cand, _gpu.scale_of(spec))
    k_max = kv.max_seq_len
    p32 = float(np.float32(0.9))
    gi, gc, gk = ssd_select_topp(r["scores"], kv.seq_lens, p32, k_max, spec.h_kv, max_len=kv.max_seq_len)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    S = r["scores"].view(-1, r["scores"].shape[-1]).cpu().numpy()
    lens = np.repeat(kv.seq_lens.cpu().numpy(), spec.h_kv)
    rows = [0, 7, 77, 130, 255]
    sub = S[rows]
    _, _, ok_k = oracle.topp(sub, lens[rows], p32, k_max)
    gk, gc, gi = gk.cpu().numpy(), gc.cpu().numpy(), gi.cpu().numpy()
    for n, rr in enumerate(rows):
        if ok_k[n] != gk[rr]:
            assert _count_ok(sub[n, :lens[rr]], p32, int(gk[rr]), k_max), (rr, int(gk[rr]), int(ok_k[n]))
    oi, oc = oracle.topk(sub, lens[rows], gk[rows], k_max)
    np.testing.assert_array_equal(gc[rows], oc)
    np.testing.assert_array_equal(gi[rows], oi)
