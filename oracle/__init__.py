"""Plain float64 CPU oracle for sparse self-speculative decoding attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` are the only callers.  The product path (the CUDA library and its
binding) never imports this package.

The arithmetic lives in ``ssd_oracle.c`` (plain loops in double precision, one
(request, KV head) unit per task on POSIX threads); this module only compiles it
with gcc and marshals numpy arrays through ctypes.  Every function states the
definition it evaluates in the C source, with the passage it follows.
"""

from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = None

F32, BF16 = 0, 1
_ERRORS = {-1: "invalid argument", -2: "page id out of range", -3: "index out of range",
           -4: "out of memory", -5: "k exceeds k_max"}


def lib_path() -> str:
    return os.path.join(_HERE, "_build", platform.machine(), "libssd_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no architecture-specific flags) and return the .so path."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(path: str):
    L = ctypes.CDLL(path)
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    L.oracle_verify.argtypes = [P, I, I64, I, I, I, P, I, P, I, P, I, I, I, D, P, P, P, P, I64, I]
    L.oracle_draft.argtypes = [P, I, I64, I, I, I, P, I, P, I, P, I, I, P, I, P, D, P, P, I]
    L.oracle_topk.argtypes = [P, I64, P, P, I, I, I, P, I, P]
    L.oracle_block_maxpool.argtypes = [P, I64, P, I, I, I, I, P, I64]
    L.oracle_block_union.argtypes = [P, P, I, I, I, P, P, P, I]
    L.oracle_block_attn.argtypes = [P, I, I64, I, I, I, P, I, P, I, P, I, I, I, P, P, I, I, D, P, P, I]
    L.oracle_kv_append.argtypes = [P, I, I64, I, I, I, P, I, P, I, I, P, P, I, P]
    L.oracle_kv_advance.argtypes = [P, P, I, I]
    L.oracle_kv_append.restype = I
    L.oracle_kv_advance.restype = I
    L.oracle_phase_assign.argtypes = [P, I, I, P]
    L.oracle_phase_flags.argtypes = [P, I, I, I64, P]
    L.oracle_phase_assign.restype = I
    L.oracle_topp_k.argtypes = [P, I64, P, D, I, I, I, I, P]
    L.oracle_topp_k.restype = I
    L.oracle_combine.argtypes = [P, P, I, I, I, P, P]
    L.oracle_combine.restype = I
    L.oracle_phase_flags.restype = I
    for fn in ("oracle_verify", "oracle_draft", "oracle_topk", "oracle_block_maxpool",
               "oracle_block_union", "oracle_block_attn"):
        getattr(L, fn).restype = ctypes.c_int
    return L


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = _load(build())
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(rc, rc)}")


def _np(x, dtype=None):
    """torch tensor / numpy array -> contiguous numpy array on the host.  bf16 tensors are
    returned as their raw uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype is not None:
        x = np.ascontiguousarray(x, dtype=dtype)
    return x


def _elem_code(arr: np.ndarray) -> int:
    if arr.dtype == np.uint16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    raise TypeError(f"unsupported element type {arr.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class PagedKV:
    """Host copy of a paged KV cache: pool [P, 2, H_kv, page_size, d], page_table [B, max_pages],
    seq_lens [B]."""

    def __init__(self, pool, page_table, seq_lens):
        self.pool = _np(pool)
        self.dtype = _elem_code(self.pool)
        self.page_table = _np(page_table, np.int32)
        self.seq_lens = _np(seq_lens, np.int32)
        P, two, self.h_kv, self.page_size, self.d = self.pool.shape
        assert two == 2
        self.num_pages = P
        self.batch, self.max_pages = self.page_table.shape

    def args(self):
        return (_ptr(self.pool), self.dtype, self.num_pages, self.page_size, self.h_kv, self.d,
                _ptr(self.page_table), self.max_pages, _ptr(self.seq_lens), self.batch)


def verify(kv: PagedKV, q, scale: float, crit_stride: int | None = None, per_candidate: bool = False,
           threads: int | None = None) -> dict:
    """Full verify attention over the paged cache.  q: [B, n_c, H_q, d].  Returns out
    [B, n_c, H_q, d], lse [B, n_c, H_q], crit [B, H_kv, stride] and, with ``per_candidate``,
    crit_cand [B, H_kv, n_c, stride] (all float64; entries t >= L_b are 0)."""
    qn = _np(q)
    B, n_c, h_q, d = qn.shape
    stride = crit_stride or max(1, int(kv.seq_lens.max()) if kv.batch else 1)
    out = np.zeros((B, n_c, h_q, d), np.float64)
    lse = np.zeros((B, n_c, h_q), np.float64)
    crit = np.zeros((B, kv.h_kv, stride), np.float64)
    cc = np.zeros((B, kv.h_kv, n_c, stride), np.float64) if per_candidate else None
    rc = _lib().oracle_verify(*kv.args(), _ptr(qn), _elem_code(qn), h_q, n_c, float(scale), _ptr(out),
                              _ptr(lse), _ptr(crit), _ptr(cc) if cc is not None else None, stride,
                              threads or default_threads())
    _check(rc, "verify")
    res = {"out": out, "lse": lse, "crit": crit}
    if cc is not None:
        res["crit_cand"] = cc
    return res


def draft(kv: PagedKV, q, idx, cnt, scale: float, threads: int | None = None) -> dict:
    """Single-query attention over the index lists.  q: [B, H_q, d]; idx [B, H_kv, k_max];
    cnt [B, H_kv].  Returns out [B, H_q, d] and lse [B, H_q] (float64)."""
    qn = _np(q)
    B, h_q, d = qn.shape
    idx_n = _np(idx, np.int32)
    cnt_n = _np(cnt, np.int32)
    k_max = idx_n.shape[-1]
    out = np.zeros((B, h_q, d), np.float64)
    lse = np.zeros((B, h_q), np.float64)
    rc = _lib().oracle_draft(*kv.args(), _ptr(qn), _elem_code(qn), h_q, _ptr(idx_n), k_max, _ptr(cnt_n),
                             float(scale), _ptr(out), _ptr(lse), threads or default_threads())
    _check(rc, "draft")
    return {"out": out, "lse": lse}


def topk(scores, lens, ks, k_max: int, rows_per_group: int = 1, len_div: int = 1):
    """Top-K per row of the fp32 score matrix [n_rows, stride].  Row r belongs to group
    r // rows_per_group, has ceil(lens[group] / len_div) entries and keeps ks[group] of them.
    Returns idx [n_rows, k_max] (ascending, -1 padded) and cnt [n_rows]."""
    s = _np(scores, np.float32)
    n_rows, stride = s.shape
    lens_n = _np(lens, np.int32)
    ks_n = _np(ks, np.int32)
    n_groups = n_rows // rows_per_group
    assert n_groups * rows_per_group == n_rows and lens_n.size == n_groups and ks_n.size == n_groups
    idx = np.zeros((n_rows, max(k_max, 1)), np.int32)[:, :k_max].copy()
    cnt = np.zeros((n_rows,), np.int32)
    rc = _lib().oracle_topk(_ptr(s), stride, _ptr(lens_n), _ptr(ks_n), n_groups, rows_per_group, len_div,
                            _ptr(idx), k_max, _ptr(cnt))
    _check(rc, "topk")
    return idx, cnt


def block_maxpool(crit_cand: np.ndarray, seq_lens, block: int, bstride: int | None = None) -> np.ndarray:
    """Max of per-candidate criticality over each ``block``-token block: [B, H_kv, n_c, n_blocks]."""
    cc = np.ascontiguousarray(crit_cand, np.float64)
    B, h_kv, n_c, stride = cc.shape
    sl = _np(seq_lens, np.int32)
    nb = bstride or max(1, (int(sl.max()) + block - 1) // block)
    out = np.full((B, h_kv, n_c, nb), -np.inf, np.float64)
    rc = _lib().oracle_block_maxpool(_ptr(cc), stride, _ptr(sl), B, h_kv, n_c, block, _ptr(out), nb)
    _check(rc, "block_maxpool")
    return out


def block_union(blocks, bcnt, umax: int | None = None):
    """Union of the candidates' block sets per unit.  blocks [U, n_c, kb], bcnt [U, n_c].
    Returns uidx [U, umax] (ascending, -1 padded), umask [U, umax] (bit i = candidate i) and
    ucnt [U]."""
    bl = _np(blocks, np.int32)
    bc = _np(bcnt, np.int32)
    U, n_c, kb = bl.shape
    um = umax or n_c * kb
    uidx = np.zeros((U, um), np.int32)
    umask = np.zeros((U, um), np.uint32)
    ucnt = np.zeros((U,), np.int32)
    rc = _lib().oracle_block_union(_ptr(bl), _ptr(bc), U, n_c, kb, _ptr(uidx), _ptr(umask), _ptr(ucnt), um)
    _check(rc, "block_union")
    return uidx, umask, ucnt


def block_attn(kv: PagedKV, q, blocks, bcnt, block: int, scale: float, threads: int | None = None) -> dict:
    """Per-candidate block-sparse attention.  q [B, n_c, H_q, d]; blocks [B, H_kv, n_c, kb];
    bcnt [B, H_kv, n_c].  Returns out [B, n_c, H_q, d] and lse [B, n_c, H_q] (float64)."""
    qn = _np(q)
    B, n_c, h_q, d = qn.shape
    bl = _np(blocks, np.int32)
    bc = _np(bcnt, np.int32)
    kb = bl.shape[-1]
    out = np.zeros((B, n_c, h_q, d), np.float64)
    lse = np.zeros((B, n_c, h_q), np.float64)
    rc = _lib().oracle_block_attn(*kv.args(), _ptr(qn), _elem_code(qn), h_q, n_c, _ptr(bl), _ptr(bc), kb,
                                  block, float(scale), _ptr(out), _ptr(lse), threads or default_threads())
    _check(rc, "block_attn")
    return {"out": out, "lse": lse}



def _use_library(path: str | None):
    """Tests only: route the wrappers through another build of the oracle source (``None``
    restores the default build).  The mutation tests use this to check that the pins catch
    planted mistakes."""
    global _LIB
    _LIB = None if path is None else _load(path)


def kv_append(pool, page_table, seq_lens, max_seq_len: int, k_new, v_new):
    """KV append (ssd_oracle.c, oracle_kv_append; reading R8): returns (new pool, written[b]).
    pool [P][2][h_kv][page][d] (float32 or bf16 bit patterns as uint16), k_new/v_new [B][n][h_kv][d]
    of the same element type.  The input pool is not modified."""
    pool = np.array(_np(pool), copy=True, order="C")
    esize = pool.dtype.itemsize
    pt = _np(page_table, np.int32)
    lens = _np(seq_lens, np.int32)
    kn = np.ascontiguousarray(_np(k_new).view(pool.dtype))
    vn = np.ascontiguousarray(_np(v_new).view(pool.dtype))
    B, n, h_kv, d = kn.shape
    ok = np.zeros(B, np.int32)
    _check(_lib().oracle_kv_append(_ptr(pool), esize, pool.shape[0], pool.shape[3], h_kv, d, _ptr(pt), pt.shape[1],
                                   _ptr(lens), B, int(max_seq_len), _ptr(kn), _ptr(vn), n, _ptr(ok)), "kv_append")
    return pool, ok


def kv_advance(seq_lens, delta, max_seq_len: int) -> np.ndarray:
    """Length advance (ssd_oracle.c, oracle_kv_advance; reading R8): seq_lens + delta where the
    result stays in [0, max_seq_len], else unchanged."""
    lens = np.array(_np(seq_lens, np.int32), copy=True)
    dl = _np(delta, np.int32)
    _check(_lib().oracle_kv_advance(_ptr(lens), _ptr(dl), lens.shape[0], int(max_seq_len)), "kv_advance")
    return lens


def phase_assign(counts, n_new: int):
    """Greedy phase-offset assignment (ssd_oracle.c, oracle_phase_assign; reading R9): returns
    (new counts, offsets of the n_new arriving requests)."""
    c = np.array(_np(counts, np.int32), copy=True)
    out = np.zeros(max(n_new, 1), np.int32)
    _check(_lib().oracle_phase_assign(_ptr(c), c.shape[0], int(n_new), _ptr(out)), "phase_assign")
    return c, out[:n_new]


def phase_flags(offsets, n_buckets: int, step: int) -> np.ndarray:
    """1 where request b verifies at `step`, else 0 (ssd_oracle.c, oracle_phase_flags; R9)."""
    off = _np(offsets, np.int32)
    out = np.zeros(max(off.shape[0], 1), np.uint8)
    _check(_lib().oracle_phase_flags(_ptr(off), off.shape[0], int(n_buckets), int(step), _ptr(out)), "phase_flags")
    return out[:off.shape[0]]


def topp(scores, lens, p: float, k_max: int, rows_per_group: int = 1, len_div: int = 1):
    """Top-p selection (ssd_oracle.c, oracle_topp_k then oracle_topk; reading R10): per row the
    smallest set of largest entries whose sum reaches p times the row total, capped at k_max.
    Returns idx [n_rows, k_max] (ascending, -1 padded), cnt [n_rows] and the per-row K."""
    s = _np(scores, np.float32)
    n_rows, stride = s.shape
    lens_n = _np(lens, np.int32)
    n_groups = n_rows // rows_per_group
    assert n_groups * rows_per_group == n_rows and lens_n.size == n_groups
    kout = np.zeros(n_rows, np.int32)
    _check(_lib().oracle_topp_k(_ptr(s), stride, _ptr(lens_n), float(p), n_groups, rows_per_group, len_div, k_max,
                                _ptr(kout)), "topp")
    idx, cnt = topk(s, np.repeat(lens_n, rows_per_group), kout, k_max, 1, len_div)
    return idx, cnt, kout


def combine(o_parts, lse_parts):
    """Split-KV combine (ssd_oracle.c, oracle_combine; SparseSpec §4.1 caches each part's LSE):
    o_parts [n_rows, n_splits, d] normalised split outputs, lse_parts [n_rows, n_splits] their
    natural-log LSEs (-inf = empty split), both float32.  Returns out [n_rows, d] =
    sum_j exp(lse_j - lse) o_j and lse [n_rows] = log sum_j exp(lse_j) (float64); a row with no
    non-empty split gives 0 and -inf."""
    o = _np(o_parts, np.float32)
    lp = _np(lse_parts, np.float32)
    n_rows, n_splits, d = o.shape
    assert lp.shape == (n_rows, n_splits)
    out = np.zeros((n_rows, d), np.float64)
    lse = np.zeros((n_rows,), np.float64)
    _check(_lib().oracle_combine(_ptr(o), _ptr(lp), n_rows, n_splits, d, _ptr(out), _ptr(lse)), "combine")
    return out, lse
