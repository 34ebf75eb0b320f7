"""ssd_draft_attn_static: the sparse draft attention entry point that allocates nothing.

Some callers cannot allocate device memory where they run the draft step: a plugin inside another
runtime that owns every device allocation and passes in only input and output buffers, or a
serving loop that must not call cudaMalloc / cudaFree (which can synchronise the device) while other
streams are busy.  For them the library keeps the draft scratch in one built-in device array.

The GPU test calls that entry point directly through the C ABI (ctypes, no Python wrapper).  Both
entry points run the same kernel on the same inputs and merge a unit's chunks in a fixed order, so
the static call must reproduce ssd_draft_attn (which takes a caller workspace) bit for bit; each
call is also checked against the CPU oracle's draft within the output tolerances of the other GPU
tests.  It makes several calls in a row with different shapes, each finding the array as the
previous one left it, and repeats the first call at the end, which must give the first call's
result bit for bit.  The host test checks that a batch too big for the array is refused before
anything runs.  The file name makes pytest collect it last.
"""

import ctypes

import pytest
import torch

import oracle

from sparse_self_speculative_verify_gb300 import KVCache, binding, ssd_draft_attn, ssd_status
from sparse_self_speculative_verify_gb300 import build as libbuild
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

DEV = "cuda:0"


def _static_call(L, kv, q, idx, cnt, scale):
    """One call of ssd_draft_attn_static; the caller (this test) owns the outputs."""
    B, h_q, d = q.shape
    out = torch.full((B, h_q, d), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, h_q), float("nan"), dtype=torch.float32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = L.ssd_draft_attn_static(kv.ref(), p(q), h_q, p(idx), idx.shape[-1], p(cnt), float(scale), p(out), p(lse),
                                 None)
    assert rc == binding.SSD_OK, L.ssd_last_error()
    return out, lse


def _case(name, over, lens, ks, k_max, seed):
    spec = W.scaled_spec(W.SPECS[name], name="na", **over)
    w = W.make_workload(spec, seed=seed, device=DEV, lengths=lens)
    idx, cnt = W.random_index_sets(w.seq_lens, spec.h_kv, torch.tensor(ks, dtype=torch.int32), k_max, seed=seed)
    return w, idx.to(DEV), cnt.to(DEV)


CALLS = [
    # (spec, overrides, lens, k per request, k_max): 7 chunks per unit, then G = 5 with an empty
    # list, then fp32 d = 64, then the first case again.
    ("qwen3_8b", dict(batch=3), [8192, 5000, 700], [410, 250, 35], 410),
    ("qwen3_8b", dict(batch=2, h_q=40), [3000, 1200], [150, 0], 150),
    ("tiny", dict(), [512, 300], [64, 40], 64),
    ("qwen3_8b", dict(batch=3), [8192, 5000, 700], [410, 250, 35], 410),
]


@pytest.mark.gpu
def test_static_matches_workspace_entry_point_on_consecutive_calls():
    _gpu.lib()
    L = binding.load()
    first = None
    for n, (name, over, lens, ks, k_max) in enumerate(CALLS):
        w, idx, cnt = _case(name, over, lens, ks, k_max, seed=7 + (n % 3))
        kv = KVCache.from_workload(w)
        q = w.q_draft[0]
        scale = _gpu.scale_of(w.spec)
        ref = ssd_draft_attn(kv, q, idx, cnt, scale)
        out, lse = _static_call(L, kv, q, idx, cnt, scale)
        torch.cuda.synchronize()
        assert ssd_status() == 0
        assert torch.equal(out, ref["out"]), f"call {n}: out differs from ssd_draft_attn"
        assert torch.equal(lse, ref["lse"]), f"call {n}: lse differs from ssd_draft_attn"
        kv_h, _ = _gpu.host_subset(w)
        oref = oracle.draft(kv_h, q.cpu(), idx.cpu(), cnt.cpu(), scale)
        _gpu.assert_out(out.cpu().numpy(), oref["out"], f"call {n} out vs oracle")
        _gpu.assert_lse(lse.cpu().numpy(), oref["lse"], f"call {n} lse vs oracle")
        if n == 0:
            first = (out.clone(), lse.clone())
        if n == len(CALLS) - 1:
            # Same inputs as the first call, after other shapes used the array: the same bits.
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), "repeat of call 0 differs"


def test_static_rejects_batches_beyond_the_builtin_scratch():
    libbuild.build()
    L = binding.load()
    kv = binding.PagedKVStruct(pool=16, dtype=binding.SSD_DTYPE_BF16, num_pages=1 << 20, page_size=16, h_kv=8, d=128,
                               page_table=256, max_pages=1024, seq_lens=512, batch=1024, max_seq_len=16384)
    need = L.ssd_draft_workspace_bytes(ctypes.byref(kv), 128, 4096)
    assert need > 16 << 20
    rc = L.ssd_draft_attn_static(ctypes.byref(kv), 4096, 128, 4096, 4096, 4096, 0.1, 8192, None, None)
    assert rc == binding.SSD_ERR_WORKSPACE
    assert b"built-in scratch" in L.ssd_last_error()
