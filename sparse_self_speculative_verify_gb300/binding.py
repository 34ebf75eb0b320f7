"""Thin Python binding of libssd (the C ABI in include/ssd.h).

Argument marshalling only: tensors are checked for device/dtype/contiguity, turned into raw
pointers and passed with torch's current CUDA stream.  Every step of the computation runs in the
CUDA kernels of libssd.so; there is no fallback.  If the library has not been built, every call
raises ``LibraryNotBuilt`` -- build it with ``sparse_self_speculative_verify_gb300.build.build()``.

PyTorch supplies device memory (outputs and zero-initialised workspaces) and streams.
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

SSD_OK, SSD_ERR_INVALID_ARG, SSD_ERR_UNSUPPORTED, SSD_ERR_WORKSPACE, SSD_ERR_CUDA, SSD_ERR_TIMEOUT = range(6)
SSD_DTYPE_F32, SSD_DTYPE_BF16 = 0, 1
FAULT_PAGE, FAULT_SEQLEN, FAULT_INDEX, FAULT_KMAX, FAULT_UNION, FAULT_TIMEOUT, FAULT_VALUE = 1, 2, 4, 8, 16, 32, 64

EXPORTED = ["ssd_last_error", "ssd_version", "ssd_status", "ssd_verify_workspace_bytes", "ssd_verify_attn",
            "ssd_verify_select", "ssd_verify_select_packed",
            "ssd_select_topk", "ssd_select_topp", "ssd_draft_workspace_bytes", "ssd_draft_attn", "ssd_draft_attn_static",
            "ssd_draft_pack_bytes", "ssd_draft_attn_packed",
            "ssd_unified_workspace_bytes", "ssd_kv_append", "ssd_kv_advance", "ssd_phase_assign", "ssd_phase_fill",
            "ssd_unified_attn", "ssd_block_union", "ssd_block_sparse_workspace_bytes", "ssd_block_sparse_attn",
            "ssd_combine"]


class LibraryNotBuilt(RuntimeError):
    pass


class SSDError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class PagedKVStruct(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("dtype", ctypes.c_int), ("num_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int), ("h_kv", ctypes.c_int), ("d", ctypes.c_int),
                ("page_table", ctypes.c_void_p), ("max_pages", ctypes.c_int), ("seq_lens", ctypes.c_void_p),
                ("batch", ctypes.c_int), ("max_seq_len", ctypes.c_int)]


_LIB = None
_LOCK = threading.Lock()


def library_path() -> str:
    return _build.lib_path()


def load(path: Optional[str] = None, as_default: bool = False):
    """Load libssd.so (no build step).  Raises LibraryNotBuilt when it is missing.  A library given
    by ``path`` serves the calls of this module only with ``as_default``."""
    global _LIB
    with _LOCK:
        if _LIB is not None and path is None:
            return _LIB
        p = path or library_path()
        if not os.path.exists(p):
            raise LibraryNotBuilt(f"{p} does not exist; build it with sparse_self_speculative_verify_gb300.build.build()")
        L = ctypes.CDLL(p)
        P, I, I64, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        KV = ctypes.POINTER(PagedKVStruct)
        sig = {
            "ssd_last_error": ([], ctypes.c_char_p),
            "ssd_version": ([], I),
            "ssd_status": ([P, ctypes.POINTER(ctypes.c_uint32)], I),
            "ssd_verify_workspace_bytes": ([KV, I, I], S),
            "ssd_verify_attn": ([KV, P, I, I, F, P, P, P, I64, P, I64, I, P, S, P], I),
            "ssd_verify_select": ([KV, P, I, I, F, P, P, P, I64, P, P, I, P, P, S, P], I),
            "ssd_verify_select_packed": ([KV, P, I, I, F, P, P, P, I64, P, P, I, P, P, S, P, S, P], I),
            "ssd_select_topk": ([P, I64, P, P, I, I, I, I, P, I, P, P], I),
            "ssd_select_topp": ([P, I64, P, F, I, I, I, I, P, I, P, P, P], I),
            "ssd_draft_workspace_bytes": ([KV, I, I], S),
            "ssd_draft_attn": ([KV, P, I, P, I, P, F, P, P, P, S, P], I),
            "ssd_draft_attn_static": ([KV, P, I, P, I, P, F, P, P, P], I),
            "ssd_draft_pack_bytes": ([KV, I], S),
            "ssd_draft_attn_packed": ([KV, P, I, P, I, P, F, P, P, P, S, I, P, S, P], I),
            "ssd_kv_append": ([KV, P, P, I, P], I),
            "ssd_kv_advance": ([P, P, I, I, P], I),
            "ssd_phase_assign": ([P, I, I, P], I),
            "ssd_phase_fill": ([P, I, I, I64, P, P], I),
            "ssd_unified_workspace_bytes": ([KV, I, I, I], S),
            "ssd_unified_attn": ([KV, P, P, P, I, I, P, I, P, F, P, P, P, I64, P, P, P, S, P], I),
            "ssd_block_union": ([P, P, I, I, I, I, P, P, P, I, P], I),
            "ssd_block_sparse_workspace_bytes": ([KV, I, I, I], S),
            "ssd_block_sparse_attn": ([KV, P, I, I, P, P, P, I, I, F, P, P, P, S, P], I),
            "ssd_combine": ([P, P, I, I, I, P, P, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        if path is None or as_default:
            _LIB = L
        return L


def _lib():
    return _LIB if _LIB is not None else load()


def _check(rc: int):
    if rc != SSD_OK:
        raise SSDError(rc, _lib().ssd_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


# ------------------------------------------------------------------------------------------------
# Paged KV cache handle and workspaces.
# ------------------------------------------------------------------------------------------------


@dataclass
class KVCache:
    """pool [num_pages, 2, h_kv, page_size, d] (bf16 or fp32), page_table [B, max_pages] int32,
    seq_lens [B] int32, max_seq_len (host int, >= every seq_len)."""
    pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    max_seq_len: int

    def __post_init__(self):
        _need(self.pool, "pool")
        _need(self.page_table, "page_table", torch.int32, self.pool.device)
        _need(self.seq_lens, "seq_lens", torch.int32, self.pool.device)
        if self.pool.dim() != 5 or self.pool.shape[1] != 2:
            raise ValueError("pool must be [num_pages, 2, h_kv, page_size, d]")
        if self.pool.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError("pool must be bf16 or fp32")
        self._struct = PagedKVStruct(
            self.pool.data_ptr(), SSD_DTYPE_BF16 if self.pool.dtype == torch.bfloat16 else SSD_DTYPE_F32,
            self.pool.shape[0], self.pool.shape[3], self.pool.shape[2], self.pool.shape[4],
            self.page_table.data_ptr(), self.page_table.shape[1], self.seq_lens.data_ptr(),
            self.seq_lens.shape[0], int(self.max_seq_len))

    @property
    def h_kv(self) -> int:
        return self.pool.shape[2]

    @property
    def d(self) -> int:
        return self.pool.shape[4]

    @property
    def batch(self) -> int:
        return self.seq_lens.shape[0]

    @property
    def device(self):
        return self.pool.device

    def ref(self):
        return ctypes.byref(self._struct)

    @classmethod
    def from_workload(cls, w) -> "KVCache":
        return cls(w.pool, w.page_table, w.seq_lens, w.max_seq_len)


class Workspace:
    """Zero-initialised device scratch buffers, grown on demand, one per (device, name).  The
    library keeps its counters in a fixed area at the start of a workspace and returns them to zero
    after each call, so a buffer is zeroed only once and serves calls of any shape in turn."""

    def __init__(self):
        self._bufs = {}

    def get(self, device, name: str, nbytes: int) -> torch.Tensor:
        key = (str(device), name)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(int(nbytes), 256) + 256, dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf

    @staticmethod
    def aligned(buf: torch.Tensor) -> int:
        p = buf.data_ptr()
        return (p + 255) & ~255


_DEFAULT_WS = Workspace()


def _ws(kv_device, name, nbytes, workspace: Optional[Workspace]):
    ws = (workspace or _DEFAULT_WS).get(kv_device, name, nbytes)
    base = Workspace.aligned(ws)
    avail = ws.data_ptr() + ws.numel() - base
    return ctypes.c_void_p(base), avail


# ------------------------------------------------------------------------------------------------
# Calls (same names as the C ABI).
# ------------------------------------------------------------------------------------------------


def ssd_version() -> int:
    return _lib().ssd_version()


def ssd_status(stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_lib().ssd_status(_stream(stream), ctypes.byref(v)))
    return v.value


def ssd_verify_attn(kv: KVCache, q: torch.Tensor, n_cand: int, scale: float, *, out=None, lse=None,
                    scores: Optional[torch.Tensor] = None, bscores: Optional[torch.Tensor] = None,
                    block_size: int = 64, want_scores: bool = True, want_lse: bool = True,
                    workspace: Optional[Workspace] = None, stream=None) -> dict:
    """Verify attention over the paged cache with fused criticality.  q [B, n_cand, h_q, d]."""
    _need(q, "q", kv.pool.dtype, kv.device)
    B, nc, h_q, d = q.shape
    assert nc == n_cand and B == kv.batch and d == kv.d
    dev = kv.device
    if out is None:
        out = torch.empty((B, nc, h_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, nc, h_q), dtype=torch.float32, device=dev)
    if scores is None and want_scores:
        scores = torch.zeros((B, kv.h_kv, max(kv.max_seq_len, 1)), dtype=torch.float32, device=dev)
    for t, n in ((out, "out"), (lse, "lse"), (scores, "scores"), (bscores, "bscores")):
        if t is not None:
            _need(t, n, torch.float32, dev)
    L = _lib()
    need = L.ssd_verify_workspace_bytes(kv.ref(), h_q, n_cand)
    wsp, avail = _ws(dev, "verify", need, workspace)
    _check(L.ssd_verify_attn(kv.ref(), _ptr(q), h_q, n_cand, float(scale), _ptr(out), _ptr(lse), _ptr(scores),
                             scores.shape[-1] if scores is not None else 0, _ptr(bscores),
                             bscores.shape[-1] if bscores is not None else 0, block_size, wsp, avail,
                             _stream(stream)))
    return {"out": out, "lse": lse, "scores": scores, "bscores": bscores}


def ssd_verify_select(kv: KVCache, q: torch.Tensor, n_cand: int, scale: float, ks: torch.Tensor, k_max: int, *,
                      out=None, lse=None, scores=None, idx=None, cnt=None, want_lse: bool = True,
                      pack: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None,
                      stream=None) -> dict:
    """Verify with the Top-K selection fused into its criticality pass.  q [B, n_cand, h_q, d];
    ks [B] int32 (K per request); idx [B * h_kv, k_max], cnt [B * h_kv].  With `pack` (a uint8 buffer
    of ssd_draft_pack_bytes(kv, k_max) bytes, 256-byte aligned), ssd_verify_select_packed: the
    selected rows are also stored there for drafts with PACK_READ."""
    _need(q, "q", kv.pool.dtype, kv.device)
    B, nc, h_q, d = q.shape
    assert nc == n_cand and B == kv.batch and d == kv.d
    dev = kv.device
    _need(ks, "ks", torch.int32, dev)
    if out is None:
        out = torch.empty((B, nc, h_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, nc, h_q), dtype=torch.float32, device=dev)
    if scores is None:
        scores = torch.zeros((B, kv.h_kv, max(kv.max_seq_len, 1)), dtype=torch.float32, device=dev)
    if idx is None:
        idx = torch.empty((B * kv.h_kv, max(k_max, 0)), dtype=torch.int32, device=dev)
    if cnt is None:
        cnt = torch.empty((B * kv.h_kv,), dtype=torch.int32, device=dev)
    for t, n, dt in ((out, "out", torch.float32), (lse, "lse", torch.float32), (scores, "scores", torch.float32),
                     (idx, "idx", torch.int32), (cnt, "cnt", torch.int32)):
        if t is not None:
            _need(t, n, dt, dev)
    L = _lib()
    need = L.ssd_verify_workspace_bytes(kv.ref(), h_q, n_cand)
    wsp, avail = _ws(dev, "verify", need, workspace)
    if pack is None:
        _check(L.ssd_verify_select(kv.ref(), _ptr(q), h_q, n_cand, float(scale), _ptr(out), _ptr(lse), _ptr(scores),
                                   scores.shape[-1], _ptr(ks), _ptr(idx), k_max, _ptr(cnt), wsp, avail,
                                   _stream(stream)))
    else:
        _need(pack, "pack", torch.uint8, dev)
        _check(L.ssd_verify_select_packed(kv.ref(), _ptr(q), h_q, n_cand, float(scale), _ptr(out), _ptr(lse),
                                          _ptr(scores), scores.shape[-1], _ptr(ks), _ptr(idx), k_max, _ptr(cnt),
                                          _ptr(pack), pack.numel(), wsp, avail, _stream(stream)))
    return {"out": out, "lse": lse, "scores": scores, "idx": idx, "cnt": cnt}


def ssd_select_topk(scores: torch.Tensor, lens: torch.Tensor, ks: torch.Tensor, k_max: int, rows_per_group: int,
                    len_div: int = 1, max_len: Optional[int] = None, *, idx=None, cnt=None, stream=None):
    """Top-K per row of a [n_rows, stride] (or [..., stride]) fp32 score tensor."""
    _need(scores, "scores", torch.float32)
    dev = scores.device
    _need(lens, "lens", torch.int32, dev)
    _need(ks, "ks", torch.int32, dev)
    stride = scores.shape[-1]
    n_rows = scores.numel() // stride
    n_groups = lens.shape[0]
    assert n_groups * rows_per_group == n_rows and ks.shape[0] == n_groups
    if max_len is None:
        max_len = stride
    if idx is None:
        idx = torch.empty((n_rows, max(k_max, 0)), dtype=torch.int32, device=dev)
    if cnt is None:
        cnt = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    _need(idx, "idx", torch.int32, dev)
    _need(cnt, "cnt", torch.int32, dev)
    _check(_lib().ssd_select_topk(_ptr(scores), stride, _ptr(lens), _ptr(ks), n_groups, rows_per_group, len_div,
                                  int(max_len), _ptr(idx), k_max, _ptr(cnt), _stream(stream)))
    return idx, cnt


def ssd_select_topp(scores: torch.Tensor, lens: torch.Tensor, p: float, k_max: int, rows_per_group: int,
                    len_div: int = 1, max_len: Optional[int] = None, *, idx=None, cnt=None, k_rows=None,
                    stream=None):
    """Top-p per row: the fewest largest entries whose sum reaches p times the row total, at most
    k_max.  Returns (idx, cnt, k_rows); k_rows is the per-row count before the Top-K pass."""
    _need(scores, "scores", torch.float32)
    dev = scores.device
    _need(lens, "lens", torch.int32, dev)
    stride = scores.shape[-1]
    n_rows = scores.numel() // stride
    n_groups = lens.shape[0]
    assert n_groups * rows_per_group == n_rows
    if max_len is None:
        max_len = stride
    if idx is None:
        idx = torch.empty((n_rows, max(k_max, 0)), dtype=torch.int32, device=dev)
    if cnt is None:
        cnt = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    if k_rows is None:
        k_rows = torch.empty((n_rows,), dtype=torch.int32, device=dev)
    for t, name in ((idx, "idx"), (cnt, "cnt"), (k_rows, "k_rows")):
        _need(t, name, torch.int32, dev)
    _check(_lib().ssd_select_topp(_ptr(scores), stride, _ptr(lens), float(p), n_groups, rows_per_group, len_div,
                                  int(max_len), _ptr(idx), k_max, _ptr(cnt), _ptr(k_rows), _stream(stream)))
    return idx, cnt, k_rows


def ssd_draft_attn(kv: KVCache, q: torch.Tensor, idx: torch.Tensor, cnt: torch.Tensor, scale: float, *, out=None,
                   lse=None, want_lse: bool = True, workspace: Optional[Workspace] = None, stream=None) -> dict:
    """Single-query attention over the selected tokens.  q [B, h_q, d]; idx [B, h_kv, k_max]."""
    _need(q, "q", kv.pool.dtype, kv.device)
    dev = kv.device
    _need(idx, "idx", torch.int32, dev)
    _need(cnt, "cnt", torch.int32, dev)
    B, h_q, d = q.shape
    k_max = idx.shape[-1]
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    L = _lib()
    need = L.ssd_draft_workspace_bytes(kv.ref(), h_q, k_max)
    wsp, avail = _ws(dev, "draft", need, workspace)
    _check(L.ssd_draft_attn(kv.ref(), _ptr(q), h_q, _ptr(idx), k_max, _ptr(cnt), float(scale), _ptr(out), _ptr(lse),
                            wsp, avail, _stream(stream)))
    return {"out": out, "lse": lse}


PACK_NONE, PACK_WRITE, PACK_READ, PACK_READ_DISCARD = 0, 1, 2, 3


def ssd_draft_pack_bytes(kv: KVCache, k_max: int) -> int:
    return int(_lib().ssd_draft_pack_bytes(kv.ref(), int(k_max)))


def ssd_draft_attn_packed(kv: KVCache, q: torch.Tensor, idx: Optional[torch.Tensor], cnt: torch.Tensor, scale: float,
                          pack: torch.Tensor, pack_mode: int, *, k_max: Optional[int] = None, out=None, lse=None,
                          want_lse: bool = True, workspace: Optional[Workspace] = None, stream=None) -> dict:
    """ssd_draft_attn with a row pack: PACK_WRITE attends through idx and stores the selected rows in
    ``pack`` (a uint8 device tensor of ssd_draft_pack_bytes bytes, 256-byte aligned); PACK_READ
    attends the rows stored by the last PACK_WRITE call (idx may be None; then k_max is required);
    PACK_READ_DISCARD reads likewise and leaves the pack undefined (the round's last draft: its lines
    leave L2 without being written back)."""
    _need(q, "q", kv.pool.dtype, kv.device)
    dev = kv.device
    if idx is not None:
        _need(idx, "idx", torch.int32, dev)
    _need(cnt, "cnt", torch.int32, dev)
    _need(pack, "pack", torch.uint8, dev)
    B, h_q, d = q.shape
    if k_max is None:
        if idx is None:
            raise ValueError("k_max is required when idx is None")
        k_max = idx.shape[-1]
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    L = _lib()
    need = L.ssd_draft_workspace_bytes(kv.ref(), h_q, k_max)
    wsp, avail = _ws(dev, "draft", need, workspace)
    _check(L.ssd_draft_attn_packed(kv.ref(), _ptr(q), h_q, _ptr(idx), int(k_max), _ptr(cnt), float(scale), _ptr(out),
                                   _ptr(lse), _ptr(pack), pack.numel(), int(pack_mode), wsp, avail, _stream(stream)))
    return {"out": out, "lse": lse}


def ssd_draft_attn_static(kv: KVCache, q: torch.Tensor, idx: torch.Tensor, cnt: torch.Tensor, scale: float, *,
                          out=None, lse=None, want_lse: bool = True, stream=None) -> dict:
    """ssd_draft_attn without a workspace: the scratch is the library's built-in device array
    (SSD_DRAFT_STATIC_SCRATCH_BYTES), so nothing is allocated for it.  For callers that cannot
    allocate device memory where they run the draft step.  Calls that can overlap on the GPU share
    that array and race; the first call on a device must come before any stream capture there."""
    _need(q, "q", kv.pool.dtype, kv.device)
    dev = kv.device
    _need(idx, "idx", torch.int32, dev)
    _need(cnt, "cnt", torch.int32, dev)
    B, h_q, d = q.shape
    k_max = idx.shape[-1]
    if out is None:
        out = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    _check(_lib().ssd_draft_attn_static(kv.ref(), _ptr(q), h_q, _ptr(idx), k_max, _ptr(cnt), float(scale), _ptr(out),
                                        _ptr(lse), _stream(stream)))
    return {"out": out, "lse": lse}


def ssd_kv_append(kv: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Writes k_new / v_new [B, n_new, h_kv, d] (the pool's dtype) at positions seq_lens[b] + j of
    every request; kv.pool is modified in place, kv.seq_lens is not."""
    _need(k_new, "k_new", kv.pool.dtype, kv.device)
    _need(v_new, "v_new", kv.pool.dtype, kv.device)
    if k_new.shape != v_new.shape or k_new.dim() != 4 or k_new.shape[0] != kv.batch or \
            k_new.shape[2] != kv.h_kv or k_new.shape[3] != kv.d:
        raise ValueError("k_new and v_new must both be [batch, n_new, h_kv, d]")
    _check(_lib().ssd_kv_append(kv.ref(), _ptr(k_new), _ptr(v_new), k_new.shape[1], _stream(stream)))


def ssd_kv_advance(seq_lens: torch.Tensor, delta: torch.Tensor, max_seq_len: int, stream=None) -> None:
    """seq_lens += delta in place on the device (results outside [0, max_seq_len] are left as they
    were and flagged in the device status)."""
    _need(seq_lens, "seq_lens", torch.int32, seq_lens.device)
    _need(delta, "delta", torch.int32, seq_lens.device)
    if delta.shape != seq_lens.shape:
        raise ValueError("delta must have the shape of seq_lens")
    _check(_lib().ssd_kv_advance(_ptr(seq_lens), _ptr(delta), seq_lens.shape[0], int(max_seq_len),
                                 _stream(stream)))


def ssd_phase_assign(counts, n_new: int):
    """Greedy phase offsets for n_new arriving requests.  counts: host int32 array [k + 1] of live
    requests per offset (numpy or CPU tensor), updated in place; returns the offsets (int32 numpy)."""
    import numpy as np
    c = counts.numpy() if isinstance(counts, torch.Tensor) else counts
    if not isinstance(c, np.ndarray) or c.dtype != np.int32 or not c.flags["C_CONTIGUOUS"]:
        raise TypeError("counts must be a contiguous int32 host array")
    out = np.zeros(max(n_new, 1), np.int32)
    _check(_lib().ssd_phase_assign(c.ctypes.data_as(ctypes.c_void_p), c.shape[0], int(n_new),
                                   out.ctypes.data_as(ctypes.c_void_p)))
    return out[:n_new]


def ssd_phase_fill(offsets: torch.Tensor, n_buckets: int, step: int, *, phase=None, stream=None) -> torch.Tensor:
    """Device phase array for ssd_unified_attn at `step`: 1 = verify, 0 = draft."""
    _need(offsets, "offsets", torch.int32, offsets.device)
    if phase is None:
        phase = torch.empty(offsets.shape, dtype=torch.uint8, device=offsets.device)
    _need(phase, "phase", torch.uint8, offsets.device)
    _check(_lib().ssd_phase_fill(_ptr(offsets), offsets.shape[0], int(n_buckets), int(step), _ptr(phase),
                                 _stream(stream)))
    return phase


def ssd_unified_attn(kv: KVCache, phase: torch.Tensor, q_verify: torch.Tensor, q_draft: torch.Tensor, n_cand: int,
                     idx: torch.Tensor, cnt: torch.Tensor, scale: float, *, out_verify=None, lse_verify=None,
                     scores=None, out_draft=None, lse_draft=None, want_scores: bool = True,
                     workspace: Optional[Workspace] = None, stream=None) -> dict:
    """Mixed batch: verify-phase requests (phase == 1) get verify + criticality, draft-phase requests
    (phase == 0) the sparse draft, in one call."""
    dev = kv.device
    _need(phase, "phase", torch.uint8, dev)
    _need(q_verify, "q_verify", kv.pool.dtype, dev)
    _need(q_draft, "q_draft", kv.pool.dtype, dev)
    _need(idx, "idx", torch.int32, dev)
    _need(cnt, "cnt", torch.int32, dev)
    B, nc, h_q, d = q_verify.shape
    k_max = idx.shape[-1]
    if out_verify is None:
        out_verify = torch.zeros((B, nc, h_q, d), dtype=torch.float32, device=dev)
    if lse_verify is None:
        lse_verify = torch.zeros((B, nc, h_q), dtype=torch.float32, device=dev)
    if scores is None and want_scores:
        scores = torch.zeros((B, kv.h_kv, max(kv.max_seq_len, 1)), dtype=torch.float32, device=dev)
    if out_draft is None:
        out_draft = torch.zeros((B, h_q, d), dtype=torch.float32, device=dev)
    if lse_draft is None:
        lse_draft = torch.zeros((B, h_q), dtype=torch.float32, device=dev)
    L = _lib()
    need = L.ssd_unified_workspace_bytes(kv.ref(), h_q, n_cand, k_max)
    wsp, avail = _ws(dev, "unified", need, workspace)
    _check(L.ssd_unified_attn(kv.ref(), _ptr(phase), _ptr(q_verify), _ptr(q_draft), h_q, n_cand, _ptr(idx), k_max,
                              _ptr(cnt), float(scale), _ptr(out_verify), _ptr(lse_verify), _ptr(scores),
                              scores.shape[-1] if scores is not None else 0, _ptr(out_draft), _ptr(lse_draft), wsp,
                              avail, _stream(stream)))
    return {"out_verify": out_verify, "lse_verify": lse_verify, "scores": scores, "out_draft": out_draft,
            "lse_draft": lse_draft}


def ssd_block_union(blocks: torch.Tensor, bcnt: torch.Tensor, nblk_max: int, umax: Optional[int] = None, *,
                    uidx=None, umask=None, ucnt=None, stream=None):
    """Union of the candidates' block sets.  blocks [units, n_cand, kb], bcnt [units, n_cand]."""
    _need(blocks, "blocks", torch.int32)
    dev = blocks.device
    _need(bcnt, "bcnt", torch.int32, dev)
    U, nc, kb = blocks.shape
    um = umax or nc * kb
    if uidx is None:
        uidx = torch.empty((U, um), dtype=torch.int32, device=dev)
    if umask is None:
        umask = torch.empty((U, um), dtype=torch.int32, device=dev)  # uint32 bit patterns
    if ucnt is None:
        ucnt = torch.empty((U,), dtype=torch.int32, device=dev)
    _need(uidx, "uidx", torch.int32, dev)
    _need(umask, "umask", torch.int32, dev)
    _need(ucnt, "ucnt", torch.int32, dev)
    assert uidx.shape == (U, um) and umask.shape == (U, um) and ucnt.shape == (U,)
    _check(_lib().ssd_block_union(_ptr(blocks), _ptr(bcnt), U, nc, kb, nblk_max, _ptr(uidx), _ptr(umask), _ptr(ucnt),
                                  um, _stream(stream)))
    return uidx, umask, ucnt


def ssd_block_sparse_attn(kv: KVCache, q: torch.Tensor, n_cand: int, uidx: torch.Tensor, umask: torch.Tensor,
                          ucnt: torch.Tensor, scale: float, block_size: int = 64, *, out=None, lse=None,
                          workspace: Optional[Workspace] = None, stream=None) -> dict:
    """Block-sparse attention of the candidates over their union blocks (each loaded once)."""
    dev = kv.device
    _need(q, "q", kv.pool.dtype, dev)
    _need(uidx, "uidx", torch.int32, dev)
    _need(umask, "umask", torch.int32, dev)
    _need(ucnt, "ucnt", torch.int32, dev)
    B, nc, h_q, d = q.shape
    umax = uidx.shape[-1]
    if out is None:
        out = torch.empty((B, nc, h_q, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, nc, h_q), dtype=torch.float32, device=dev)
    L = _lib()
    need = L.ssd_block_sparse_workspace_bytes(kv.ref(), h_q, n_cand, umax)
    wsp, avail = _ws(dev, "block", need, workspace)
    _check(L.ssd_block_sparse_attn(kv.ref(), _ptr(q), h_q, n_cand, _ptr(uidx), _ptr(umask), _ptr(ucnt), umax,
                                   block_size, float(scale), _ptr(out), _ptr(lse), wsp, avail, _stream(stream)))
    return {"out": out, "lse": lse}


def ssd_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, *, out=None, lse=None, stream=None):
    """LSE merge of split partials: o_parts [rows, splits, d], lse_parts [rows, splits]."""
    _need(o_parts, "o_parts", torch.float32)
    dev = o_parts.device
    _need(lse_parts, "lse_parts", torch.float32, dev)
    R, S, d = o_parts.shape
    if out is None:
        out = torch.empty((R, d), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((R,), dtype=torch.float32, device=dev)
    _check(_lib().ssd_combine(_ptr(o_parts), _ptr(lse_parts), R, S, d, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse
