"""Helpers for the GPU parity tests: host copies of (sub)workloads for the oracle, and the
comparisons with the parity tolerances (outputs: max |diff| <= 2e-3; criticality:
|diff| <= 1e-3 |ref| + 1e-6; indices: bit-exact when both sides select from the same fp32 scores)."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from sparse_self_speculative_verify_gb300 import build as libbuild
from sparse_self_speculative_verify_gb300 import binding

OUT_TOL = 2e-3
LSE_TOL = 2e-3
SCORE_RTOL = 1e-3
SCORE_ATOL = 1e-6

_built = False


def lib():
    global _built
    if not _built:
        libbuild.build()
        binding.load()
        _built = True


def scale_of(spec) -> float:
    return 1.0 / math.sqrt(spec.d)


def host_subset(w, reqs=None):
    """Oracle view of requests ``reqs`` of a device workload: their pages gathered into a compact
    host pool with a remapped page table (layout only)."""
    B = w.spec.batch
    reqs = list(range(B)) if reqs is None else list(reqs)
    ps = w.spec.page_size
    lens = w.seq_lens.cpu()[reqs]
    pt = w.page_table.cpu()[reqs]
    npg = [(int(L) + ps - 1) // ps for L in lens.tolist()]
    pages = torch.cat([pt[i, :n] for i, n in enumerate(npg)]).to(torch.int64)
    pool = w.pool[pages.to(w.pool.device)].cpu()
    new_pt = torch.full((len(reqs), max(1, max(npg))), -1, dtype=torch.int32)
    off = 0
    for i, n in enumerate(npg):
        new_pt[i, :n] = torch.arange(off, off + n, dtype=torch.int32)
        off += n
    kv = oracle.PagedKV(pool, new_pt, lens)
    return kv, reqs


def max_abs(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    return float(np.nanmax(np.abs(a - b))) if not (np.isnan(a).any() or np.isnan(b).any()) else float("inf")


def assert_out(got, ref, what="out", tol=OUT_TOL):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = max_abs(got, ref)
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol}"
    return err


def assert_lse(got, ref, what="lse"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: -inf pattern differs"
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= LSE_TOL, f"{what}: max abs error {err:.3e}"


def assert_scores(got, ref, lens, what="scores"):
    """got/ref [B, H_kv, >= L]; only t < L_b is compared."""
    worst = 0.0
    for b, L in enumerate(lens):
        g = np.asarray(got[b, :, :L], np.float64)
        r = np.asarray(ref[b, :, :L], np.float64)
        assert np.isfinite(g).all(), f"{what}: request {b}: non-finite scores"
        d = np.abs(g - r)
        lim = SCORE_RTOL * np.abs(r) + SCORE_ATOL
        bad = d > lim
        assert not bad.any(), f"{what}: request {b}: {int(bad.sum())} entries off, worst {float((d - lim).max()):.3e}"
        worst = max(worst, float((d / lim).max()) if d.size else 0.0)
    return worst


def assert_valid_topk(idx, cnt, ref_scores, ks, lens, rows_per_group):
    """idx (one row per (b, g)) is a valid top-K of the float64 reference scores within the score
    tolerance: every kept score >= every dropped score minus the tolerance, ascending, distinct."""
    idx = np.asarray(idx)
    n_rows = idx.shape[0]
    for r in range(n_rows):
        b = r // rows_per_group
        L = int(lens[b])
        K = min(int(ks[b]), L)
        assert int(cnt[r]) == K
        sel = idx[r, :K]
        assert (np.diff(sel) > 0).all() and (sel >= 0).all() and (sel < L).all()
        s = np.asarray(ref_scores[r][:L], np.float64)
        keep = np.zeros(L, bool)
        keep[sel] = True
        if K == 0 or K == L:
            continue
        tol = SCORE_RTOL * np.abs(s) + SCORE_ATOL
        lo_kept = float((s[keep] + tol[keep]).min())
        hi_drop = float((s[~keep] - tol[~keep]).max())
        assert lo_kept >= hi_drop, f"row {r}: kept {lo_kept} < dropped {hi_drop}"
