"""Device-side bounds checks: bad inputs are skipped (zero-filled) and reported in the status
word; nothing traps and the context stays usable."""

import pytest
import torch

from sparse_self_speculative_verify_gb300 import (KVCache, binding, ssd_draft_attn, ssd_status,
                                                 ssd_verify_attn)
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _w():
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="f", batch=2)
    return W.make_workload(spec, seed=1, device=DEV, lengths=[300, 200])


def test_bad_page_id_sets_fault():
    _gpu.lib()
    w = _w()
    pt = w.page_table.clone()
    pt[0, 3] = w.num_pages + 1000  # outside the pool
    kv = KVCache(w.pool, pt, w.seq_lens, w.max_seq_len)
    ssd_verify_attn(kv, w.q_verify, w.spec.n_cand, 0.1)
    assert ssd_status() & binding.FAULT_PAGE
    assert ssd_status() == 0  # cleared by the read


def test_seq_len_above_max_sets_fault():
    _gpu.lib()
    w = _w()
    kv = KVCache(w.pool, w.page_table, w.seq_lens, 250)  # request 0 holds 300 > 250
    ssd_verify_attn(kv, w.q_verify, w.spec.n_cand, 0.1)
    assert ssd_status() & binding.FAULT_SEQLEN


def test_draft_index_out_of_range_sets_fault():
    _gpu.lib()
    w = _w()
    kv = KVCache.from_workload(w)
    idx = torch.zeros((2, w.spec.h_kv, 4), dtype=torch.int32, device=DEV)
    idx[1, 0, 2] = 250  # >= L = 200
    cnt = torch.full((2, w.spec.h_kv), 4, dtype=torch.int32, device=DEV)
    ssd_draft_attn(kv, w.q_draft[0], idx, cnt, 0.1)
    assert ssd_status() & binding.FAULT_INDEX
    # The context is still usable.
    r = ssd_verify_attn(kv, w.q_verify, w.spec.n_cand, 0.1)
    torch.cuda.synchronize()
    assert torch.isfinite(r["out"]).all()
    assert ssd_status() == 0


def test_host_side_errors_raise():
    _gpu.lib()
    w = _w()
    kv = KVCache.from_workload(w)
    with pytest.raises(binding.SSDError) as e:
        ssd_verify_attn(kv, w.q_verify[:, :, :7].contiguous(), w.spec.n_cand, 0.1)  # h_q not a multiple of h_kv
    assert e.value.code == binding.SSD_ERR_INVALID_ARG
