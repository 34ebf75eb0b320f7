"""KV append and length advance on the GPU against the CPU oracle (bit-exact: these are copies)."""

import numpy as np
import pytest
import torch

import oracle
from sparse_self_speculative_verify_gb300 import (KVCache, ssd_kv_advance, ssd_kv_append, ssd_status,
                                                 ssd_verify_attn)
from sparse_self_speculative_verify_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _extended(w, n_new, extra_max=0):
    """The workload's cache with pages allocated (from its spare pages) for n_new more tokens per
    request; max_seq_len covers them plus extra_max."""
    ps = w.spec.page_size
    lens = w.seq_lens.cpu().tolist()
    need = [(L + n_new + ps - 1) // ps for L in lens]
    old = w.page_table.cpu()
    pt = torch.full((len(lens), max(need) + 1), -1, dtype=torch.int32)
    pt[:, :old.shape[1]] = old
    used = set(old[old >= 0].tolist())
    spare = [p for p in range(w.pool.shape[0]) if p not in used]
    k = 0
    for b, L in enumerate(lens):
        for j in range((L + ps - 1) // ps, need[b]):
            pt[b, j] = spare[k]
            k += 1
    max_len = max(L + n_new for L in lens) + extra_max
    return KVCache(w.pool, pt.to(DEV), w.seq_lens.clone(), max_len)


def _rand_new(spec, B, n, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    mk = lambda: torch.randn((B, n, spec.h_kv, spec.d), generator=g).to(dt).to(DEV)  # noqa: E731
    return mk(), mk()


CASES = [("qwen3_8b", dict(batch=3), [700, 129, 2048], 5), ("tiny", dict(d=64), [300, 17], 7),
         ("qwen3_8b", dict(batch=2, page_size=64), [64, 1000], 16)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{'_'.join(map(str, c[2]))}-n{c[3]}")
def test_append_matches_oracle(case):
    _gpu.lib()
    name, over, lens, n = case
    spec = W.scaled_spec(W.SPECS[name], name="kv", **over)
    w = W.make_workload(spec, seed=61, device=DEV, lengths=lens, spare_pages=64)
    kv = _extended(w, n)
    k_new, v_new = _rand_new(spec, len(lens), n, 3)
    before = kv.pool.clone()
    want, ok = oracle.kv_append(before, kv.page_table, kv.seq_lens, kv.max_seq_len, k_new, v_new)
    ssd_kv_append(kv, k_new, v_new)
    torch.cuda.synchronize()
    assert ssd_status() == 0
    assert ok.all()
    got = oracle._np(kv.pool)
    np.testing.assert_array_equal(got.view(np.uint8), want.view(np.uint8))
    assert kv.seq_lens.cpu().tolist() == lens


def test_append_skips_bad_requests_like_the_oracle():
    _gpu.lib()
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="kvs", batch=3)
    lens, n = [500, 300, 200], 6
    w = W.make_workload(spec, seed=67, device=DEV, lengths=lens, spare_pages=16)
    kv = _extended(w, n)
    kv = KVCache(kv.pool, kv.page_table, kv.seq_lens, 504)  # request 0 would end at 506 > 504
    pt = kv.page_table.cpu()
    pt[2, (lens[2] + n - 1) // spec.page_size] = -1  # request 2's last new token has no page
    kv = KVCache(kv.pool, pt.to(DEV), kv.seq_lens, kv.max_seq_len)
    k_new, v_new = _rand_new(spec, 3, n, 5)
    want, ok = oracle.kv_append(kv.pool, kv.page_table, kv.seq_lens, kv.max_seq_len, k_new, v_new)
    ssd_kv_append(kv, k_new, v_new)
    torch.cuda.synchronize()
    st = ssd_status()
    assert st & _gpu.binding.FAULT_SEQLEN and st & _gpu.binding.FAULT_PAGE
    assert ok.tolist() == [0, 1, 0]
    np.testing.assert_array_equal(oracle._np(kv.pool).view(np.uint8), want.view(np.uint8))


def test_advance_matches_oracle_and_flags_out_of_range():
    _gpu.lib()
    lens = torch.tensor([5, 9, 0, 12, 7], dtype=torch.int32, device=DEV)
    delta = torch.tensor([3, -9, -1, 1, -2], dtype=torch.int32, device=DEV)
    want = oracle.kv_advance(lens, delta, 12)
    ssd_kv_advance(lens, delta, 12)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == want.tolist() == [8, 0, 0, 12, 5]
    assert ssd_status() & _gpu.binding.FAULT_SEQLEN


def test_round_append_advance_verify_rollback():
    """Candidates appended and the lengths advanced: verify over the grown cache matches the oracle
    on the oracle's appended cache; accepting a of n_c candidates rolls the lengths back to
    L + a."""
    _gpu.lib()
    spec = W.scaled_spec(W.SPECS["qwen3_8b"], name="kvr", batch=2)
    lens, n_c = [900, 333], spec.n_cand
    w = W.make_workload(spec, seed=71, device=DEV, lengths=lens, spare_pages=8)
    kv = _extended(w, n_c)
    k_new, v_new = _rand_new(spec, 2, n_c, 7)
    want_pool, _ = oracle.kv_append(kv.pool, kv.page_table, kv.seq_lens, kv.max_seq_len, k_new, v_new)
    ssd_kv_append(kv, k_new, v_new)
    ssd_kv_advance(kv.seq_lens, torch.full((2,), n_c, dtype=torch.int32, device=DEV), kv.max_seq_len)
    r = ssd_verify_attn(kv, w.q_verify, n_c, _gpu.scale_of(spec))
    torch.cuda.synchronize()
    assert ssd_status() == 0
    grown = [L + n_c for L in lens]
    assert kv.seq_lens.cpu().tolist() == grown
    ref = oracle.verify(oracle.PagedKV(want_pool, kv.page_table, np.array(grown, np.int32)), w.q_verify.cpu(),
                        _gpu.scale_of(spec), crit_stride=kv.max_seq_len)
    _gpu.assert_out(r["out"].cpu().numpy(), ref["out"], "verify after append")
    _gpu.assert_scores(r["scores"].cpu().numpy(), ref["crit"], grown)
    accepted = torch.tensor([2, n_c], dtype=torch.int32, device=DEV)
    ssd_kv_advance(kv.seq_lens, accepted - n_c, kv.max_seq_len)
    torch.cuda.synchronize()
    assert kv.seq_lens.cpu().tolist() == [lens[0] + 2, lens[1] + n_c]
