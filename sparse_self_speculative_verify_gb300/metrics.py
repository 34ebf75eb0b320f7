"""Byte and FLOP accounting of the hot path (algorithmic work, independent of the implementation).

Units: one (token, KV head) of the cache is 2 * d * elem_bytes bytes of K and V (512 B at d = 128
in bf16).  Verify reads every token of every request once; each draft reads the selected tokens;
select reads 4 bytes of score per token.
"""

from __future__ import annotations


def kv_bytes_per_token_head(d: int, elem_bytes: int) -> int:
    return 2 * d * elem_bytes


def kv_bytes_per_token(h_kv: int, d: int, elem_bytes: int, layers: int = 1) -> int:
    """K+V bytes one token adds to the cache of a model with ``layers`` attention layers."""
    return layers * h_kv * kv_bytes_per_token_head(d, elem_bytes)


def verify_kv_bytes(seq_lens, h_kv: int, d: int, elem_bytes: int) -> int:
    return int(sum(int(L) for L in seq_lens)) * h_kv * kv_bytes_per_token_head(d, elem_bytes)


def draft_kv_bytes(k_per_req, seq_lens, h_kv: int, d: int, elem_bytes: int) -> int:
    sel = sum(min(int(k), int(L)) for k, L in zip(k_per_req, seq_lens))
    return int(sel) * h_kv * kv_bytes_per_token_head(d, elem_bytes)


def verify_call_bytes(seq_lens, batch: int, h_q: int, h_kv: int, d: int, elem_bytes: int, n_cand: int,
                      scores: bool = True) -> int:
    """Algorithmic HBM bytes of one ssd_verify_attn call: KV, queries, outputs (fp32), LSE, and the
    fp32 criticality row written for every token."""
    tok = int(sum(int(L) for L in seq_lens))
    b = tok * h_kv * kv_bytes_per_token_head(d, elem_bytes)
    b += batch * n_cand * h_q * d * elem_bytes  # q
    b += batch * n_cand * h_q * (d + 1) * 4  # out + lse
    if scores:
        b += tok * h_kv * 4
    return b


def verify_flops(seq_lens, h_q: int, d: int, n_cand: int) -> int:
    """QK^T and PV multiply-adds of the visible (row, token) pairs, 2 flops each."""
    total = 0
    for L in seq_lens:
        L = int(L)
        vis = sum(L - n_cand + i + 1 for i in range(n_cand))
        total += vis * h_q * d * 2 * 2
    return total


def round_kv_bytes(seq_lens, k_per_req, h_kv: int, d: int, elem_bytes: int, k: int) -> int:
    """KV bytes of one speculative round of one layer: a verify plus k drafts."""
    return verify_kv_bytes(seq_lens, h_kv, d, elem_bytes) + k * draft_kv_bytes(k_per_req, seq_lens, h_kv, d,
                                                                                elem_bytes)
