"""Greedy phase assignment for the unified batch (host function, exact) and the per-step phase
array (GPU), against the CPU oracle; then a unified launch fed by the greedy phases."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import binding, ssd_phase_assign, ssd_phase_fill, ssd_status
from sparse_self_speculative_verify_gb300 import build as libbuild
from sparse_self_speculative_verify_gb300 import workloads as W

DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load()


def test_phase_assign_matches_oracle(lib):
    rng = np.random.default_rng(3)
    for nb in (1, 2, 5, 9):
        for _ in range(20):
            counts = rng.integers(0, 6, nb).astype(np.int32)
            n_new = int(rng.integers(0, 30))
            want_c, want_o = oracle.phase_assign(counts, n_new)
            got_o = ssd_phase_assign(counts, n_new)  # updates counts in place
            assert got_o.tolist() == want_o.tolist()
            assert counts.tolist() == want_c.tolist()


def test_phase_assign_argument_errors(lib):
    import ctypes
    E = binding.SSD_ERR_INVALID_ARG
    c = np.zeros(3, np.int32)
    p = c.ctypes.data_as(ctypes.c_void_p)
    assert lib.ssd_phase_assign(None, 3, 1, p) == E
    assert lib.ssd_phase_assign(p, 0, 1, p) == E
    assert lib.ssd_phase_assign(p, 3, 2, None) == E
    assert lib.ssd_phase_fill(None, 4, 5, 0, None, None) == E
    assert lib.ssd_phase_fill(None, 0, 5, 0, None, None) == binding.SSD_OK  # empty batch: no launch
    assert lib.ssd_phase_fill(p, 4, 0, 0, p, None) == E


@pytest.mark.gpu
def test_phase_fill_matches_oracle(lib):
    rng = np.random.default_rng(5)
    nb = 5
    offs = rng.integers(0, nb, 1000).astype(np.int32)
    d_off = torch.from_numpy(offs).to(DEV)
    for step in (0, 1, 4, 7, 123456789):
        got = ssd_phase_fill(d_off, nb, step).cpu().numpy()
        assert got.tolist() == oracle.phase_flags(offs, nb, step).tolist()
    assert ssd_status() == 0
    bad = d_off.clone()
    bad[3] = nb
    got = ssd_phase_fill(bad, nb, 0).cpu().numpy()
    assert got[3] == 0 and ssd_status() & binding.FAULT_INDEX


@pytest.mark.gpu
def test_unified_launch_with_greedy_phases(lib):
    """B requests arrive into empty buckets; at every step of one round exactly the requests of one
    bucket verify, and the unified launch on that phase array matches the oracle."""
    from tests.test_gpu_unified import _run_and_check
    spec = W.scaled_spec(W.SPECS["qwen3_14b_unified"], name="unig", batch=10, len_lo=600, len_hi=4096,
                         len_median=2000.0)
    w = W.make_workload(spec, seed=9, device=DEV)
    nb = spec.k + 1
    offs = ssd_phase_assign(np.zeros(nb, np.int32), spec.batch)
    d_off = torch.from_numpy(offs).to(DEV)
    seen = np.zeros(spec.batch, np.int64)
    for step in range(nb):
        ph = ssd_phase_fill(d_off, nb, step).cpu().numpy()
        seen += ph
        assert len(set(offs[ph == 1].tolist())) == 1
    assert seen.tolist() == [1] * spec.batch
    step = next(s for s in range(nb) if 0 < ssd_phase_fill(d_off, nb, s).sum().item() < spec.batch)
    _run_and_check(dataclasses.replace(w, phase=ssd_phase_fill(d_off, nb, step)))
