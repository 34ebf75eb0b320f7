"""The C-ABI library loads, exports every function include/ssd.h declares, and rejects bad
arguments on the host (no kernel is launched by these calls)."""

import ctypes
import os
import re

import pytest

from sparse_self_speculative_verify_gb300 import binding
from sparse_self_speculative_verify_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.ssd_version() == 0x10000


def _kv(**over):
    d = dict(pool=16, dtype=binding.SSD_DTYPE_BF16, num_pages=10, page_size=16, h_kv=8, d=128, page_table=256,
             max_pages=4, seq_lens=512, batch=2, max_seq_len=64)
    d.update(over)
    return binding.PagedKVStruct(**d)


def test_workspace_queries(lib):
    kv = _kv()
    vb = lib.ssd_verify_workspace_bytes(ctypes.byref(kv), 32, 5)
    assert vb > 0 and vb % 256 == 0
    kv2 = _kv(max_seq_len=1024, max_pages=64)
    assert lib.ssd_verify_workspace_bytes(ctypes.byref(kv2), 32, 5) > vb
    assert lib.ssd_verify_workspace_bytes(None, 32, 5) == 0
    assert lib.ssd_draft_workspace_bytes(ctypes.byref(kv), 32, 410) > lib.ssd_draft_workspace_bytes(ctypes.byref(kv), 32, 64)
    assert lib.ssd_unified_workspace_bytes(ctypes.byref(kv), 32, 5, 64) >= vb
    assert lib.ssd_block_sparse_workspace_bytes(ctypes.byref(kv), 32, 5, 80) > 0


CASES = [
    ("null kv", dict(kv=None), binding.SSD_ERR_INVALID_ARG),
    ("bad dtype", dict(kvo=dict(dtype=7)), binding.SSD_ERR_UNSUPPORTED),
    ("bad head dim", dict(kvo=dict(d=96)), binding.SSD_ERR_UNSUPPORTED),
    ("page size not pow2", dict(kvo=dict(page_size=12)), binding.SSD_ERR_UNSUPPORTED),
    ("max_seq_len > pages", dict(kvo=dict(max_seq_len=65)), binding.SSD_ERR_INVALID_ARG),
    ("unaligned pool", dict(kvo=dict(pool=24)), binding.SSD_ERR_INVALID_ARG),
    ("h_q not multiple", dict(h_q=30), binding.SSD_ERR_INVALID_ARG),
    ("too many rows", dict(h_q=128, n_cand=5), binding.SSD_ERR_UNSUPPORTED),
    ("null q", dict(q=None), binding.SSD_ERR_INVALID_ARG),
    ("short workspace", dict(ws_bytes=100), binding.SSD_ERR_WORKSPACE),
    ("scores stride", dict(scores=4096, scores_stride=10), binding.SSD_ERR_INVALID_ARG),
    ("block size", dict(bscores=4096, bscores_stride=4, block_size=32), binding.SSD_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("name,over,code", CASES, ids=[c[0] for c in CASES])
def test_verify_argument_errors(lib, name, over, code):
    kv = _kv(**over.get("kvo", {}))
    kvp = None if "kv" in over and over["kv"] is None else ctypes.byref(kv)
    ws_bytes = over.get("ws_bytes", 1 << 40)
    rc = lib.ssd_verify_attn(kvp, over.get("q", 4096), over.get("h_q", 32), over.get("n_cand", 5), 0.1, 8192, None,
                             over.get("scores"), over.get("scores_stride", 0), over.get("bscores"),
                             over.get("bscores_stride", 0), over.get("block_size", 64), 1 << 20, ws_bytes, None)
    assert rc == code, lib.ssd_last_error()
    assert lib.ssd_last_error()


def test_verify_select_argument_errors(lib):
    kv = _kv()
    E = binding.SSD_ERR_INVALID_ARG

    def call(**o):
        return lib.ssd_verify_select(ctypes.byref(kv), 4096, 32, 5, 0.1, 8192, None, o.get("scores", 4096),
                                     o.get("stride", 1 << 16), o.get("ks", 64), o.get("idx", 128), o.get("k_max", 4),
                                     o.get("cnt", 256), 1 << 20, 1 << 40, None)
    for over in (dict(ks=None), dict(scores=None), dict(cnt=None), dict(idx=None), dict(k_max=-1), dict(stride=1)):
        assert call(**over) == E, (over, lib.ssd_last_error())


def test_select_argument_errors(lib):
    assert lib.ssd_select_topk(None, 10, 1, 1, 1, 1, 1, 10, 1, 4, 1, None) == binding.SSD_ERR_INVALID_ARG
    assert lib.ssd_select_topk(4096, 5, 16, 16, 1, 1, 1, 10, 64, 4, 64, None) == binding.SSD_ERR_INVALID_ARG
    assert lib.ssd_select_topk(4096, 10, 16, 16, 1, 0, 1, 10, 64, 4, 64, None) == binding.SSD_ERR_INVALID_ARG
    # Zero rows: nothing to do, no device work.
    assert lib.ssd_select_topk(4096, 10, 16, 16, 0, 1, 1, 10, 64, 4, 64, None) == binding.SSD_OK


def test_select_topp_argument_errors(lib):
    E = binding.SSD_ERR_INVALID_ARG
    # scores, stride, lens, p, n_groups, rows_per_group, len_div, max_len, idx, k_max, cnt, k_rows
    assert lib.ssd_select_topp(4096, 10, 16, 0.5, 1, 1, 1, 10, 64, 4, 64, None, None) == E  # k_rows NULL
    for bad_p in (-0.25, 1.25, float("nan")):
        assert lib.ssd_select_topp(4096, 10, 16, bad_p, 1, 1, 1, 10, 64, 4, 64, 128, None) == E
    assert lib.ssd_select_topp(4096, 5, 16, 0.5, 1, 1, 1, 10, 64, 4, 64, 128, None) == E  # stride < max_len
    assert lib.ssd_select_topp(4096, 10, 16, 0.5, 1, 1, 0, 10, 64, 4, 64, 128, None) == E  # len_div 0
    assert lib.ssd_select_topp(4096, 10, 16, 0.5, 0, 1, 1, 10, 64, 4, 64, 128, None) == binding.SSD_OK


def test_draft_and_union_argument_errors(lib):
    kv = _kv()
    assert lib.ssd_draft_attn(ctypes.byref(kv), None, 32, 16, 8, 16, 0.1, 16, None, 1 << 20, 1 << 40,
                              None) == binding.SSD_ERR_INVALID_ARG
    assert lib.ssd_draft_attn(ctypes.byref(kv), 16, 8 * 17, 16, 8, 16, 0.1, 16, None, 1 << 20, 1 << 40,
                              None) == binding.SSD_ERR_UNSUPPORTED  # group of 17 heads
    assert lib.ssd_block_union(16, 16, 4, 33, 16, 2048, 16, 16, 16, 80, None) == binding.SSD_ERR_UNSUPPORTED
    assert lib.ssd_combine(None, 16, 4, 2, 128, 16, None, None) == binding.SSD_ERR_INVALID_ARG


def test_draft_pack_sizes_and_argument_errors(lib):
    kv = _kv()
    need = lib.ssd_draft_pack_bytes(ctypes.byref(kv), 410)
    assert need == 2 * 8 * 7 * 2 * 64 * 128 * 2  # units x chunks x (K, V) x 64 rows x d x bf16
    assert lib.ssd_draft_pack_bytes(ctypes.byref(_kv(dtype=binding.SSD_DTYPE_F32)), 64) == 2 * 8 * 2 * 64 * 128 * 4
    assert lib.ssd_draft_pack_bytes(None, 4) == 0
    assert lib.ssd_draft_pack_bytes(ctypes.byref(_kv(d=96)), 4) == 0
    E, W = binding.SSD_ERR_INVALID_ARG, binding.SSD_ERR_WORKSPACE

    def call(idx, pack, pack_bytes, mode):
        return lib.ssd_draft_attn_packed(ctypes.byref(kv), 16, 32, idx, 410, 16, 0.1, 16, None, pack, pack_bytes, mode,
                                         1 << 20, 1 << 40, None)
    assert call(16, 1 << 21, need, 4) == E            # unknown mode (3 is SSD_PACK_READ_DISCARD)
    assert call(None, 1 << 21, need, 1) == E          # writing the pack reads idx
    assert call(16, 1 << 21, need - 1, 1) == W        # pack too small
    assert call(None, None, need, 2) == W             # no pack to read
    assert call(None, (1 << 21) + 16, need, 2) == E   # pack not 256-byte aligned


def test_kv_append_and_advance_argument_errors(lib):
    kv = _kv()
    E, OK = binding.SSD_ERR_INVALID_ARG, binding.SSD_OK
    assert lib.ssd_kv_append(ctypes.byref(kv), None, 4096, 2, None) == E  # no k_new
    assert lib.ssd_kv_append(ctypes.byref(kv), 4096, 4096, -1, None) == E  # negative count
    assert lib.ssd_kv_append(ctypes.byref(kv), 4104, 4096, 2, None) == E  # k_new not 16-byte aligned
    assert lib.ssd_kv_append(None, 4096, 4096, 2, None) == E
    assert lib.ssd_kv_append(ctypes.byref(kv), 4096, 4096, 0, None) == OK  # nothing to append, no launch
    assert lib.ssd_kv_advance(None, 4096, 4, 100, None) == E
    assert lib.ssd_kv_advance(4096, 4096, -1, 100, None) == E
    assert lib.ssd_kv_advance(4096, 4096, 0, 100, None) == OK  # empty batch, no launch


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(binding.LibraryNotBuilt):
        binding.load(str(tmp_path / "missing.so"))
