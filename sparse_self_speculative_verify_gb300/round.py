"""One speculative round on one attention layer: verify (with criticality) -> Top-K select -> k
sparse drafts, with every buffer allocated once so the round can be replayed or captured in a CUDA
graph.

SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
Sparse Attention") §4.1: the sparse pattern is refreshed by every verify and stays fixed for the k
drafts that follow it (the refresh stride equals k); §2.3 / §3.2: a round is k drafts plus one
verify of the k+1 positions.
"""

from __future__ import annotations

import math
from contextlib import nullcontext as _nullcontext
from typing import Optional

import torch

from . import binding as B


class SpecRound:
    def __init__(self, kv: B.KVCache, h_q: int, n_cand: int, k_max: int, scale: Optional[float] = None,
                 workspace: Optional[B.Workspace] = None, pack_rows: bool = True, pack_in_select: bool = False):
        self.kv = kv
        self.h_q = h_q
        self.n_cand = n_cand
        self.k_max = k_max
        self.scale = scale if scale is not None else 1.0 / math.sqrt(kv.d)
        dev = kv.device
        Bsz, hkv, d = kv.batch, kv.h_kv, kv.d
        self.ws = workspace or B.Workspace()
        self.out_v = torch.empty((Bsz, n_cand, h_q, d), dtype=torch.float32, device=dev)
        self.lse_v = torch.empty((Bsz, n_cand, h_q), dtype=torch.float32, device=dev)
        self.scores = torch.zeros((Bsz, hkv, max(kv.max_seq_len, 1)), dtype=torch.float32, device=dev)
        self.idx = torch.empty((Bsz * hkv, k_max), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((Bsz * hkv,), dtype=torch.int32, device=dev)
        self.out_d = torch.empty((Bsz, h_q, d), dtype=torch.float32, device=dev)
        self.lse_d = torch.empty((Bsz, h_q), dtype=torch.float32, device=dev)
        # Row pack: the selected K / V rows stored contiguously, by the first draft after a selection
        # or (pack_in_select) by the fused verify-select itself; the other drafts of the round read
        # them from there.  On the Qwen3-8B round the first draft's gather is the cheaper of the two
        # (the criticality pass's copy lengthens the verify call by more than it saves the draft).
        self.pack_in_select = pack_in_select
        self.pack = None
        if pack_rows:
            n = B.ssd_draft_pack_bytes(kv, k_max)
            self.pack = torch.empty(n + 256, dtype=torch.uint8, device=dev)
            off = (-self.pack.data_ptr()) % 256
            self.pack = self.pack[off:off + n]
        self._packed = False

    def verify(self, q_verify: torch.Tensor, stream=None):
        return B.ssd_verify_attn(self.kv, q_verify, self.n_cand, self.scale, out=self.out_v, lse=self.lse_v,
                                 scores=self.scores, workspace=self.ws, stream=stream)

    def verify_select(self, q_verify: torch.Tensor, k_per_req: torch.Tensor, stream=None):
        """verify + select in one call: the selection runs inside the criticality pass, which also
        stores the selected rows in the row pack (pack_in_select), so every draft reads it."""
        pack = self.pack if self.pack_in_select else None
        r = B.ssd_verify_select(self.kv, q_verify, self.n_cand, self.scale, k_per_req, self.k_max, out=self.out_v,
                                lse=self.lse_v, scores=self.scores, idx=self.idx, cnt=self.cnt, pack=pack,
                                workspace=self.ws, stream=stream)
        self._packed = pack is not None
        return r

    def select(self, k_per_req: torch.Tensor, stream=None):
        self._packed = False
        return B.ssd_select_topk(self.scores, self.kv.seq_lens, k_per_req, self.k_max, self.kv.h_kv,
                                 max_len=self.kv.max_seq_len, idx=self.idx, cnt=self.cnt, stream=stream)

    def set_selection(self, idx: torch.Tensor, cnt: torch.Tensor, stream=None):
        """Install a selection made elsewhere (idx [B, H_kv, k_max] int32, cnt [B, H_kv]) in place
        of the last select's; the next draft stores the row pack again."""
        self._packed = False
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            self.idx.view(self.kv.batch, self.kv.h_kv, self.k_max).copy_(idx)
            self.cnt.view(self.kv.batch, self.kv.h_kv).copy_(cnt)

    def draft(self, q_draft: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None, last: bool = False):
        """One draft over the current selection.  With the row pack, the first draft after a select
        stores the selected rows and the following ones read them (same results within the oracle
        tolerance).  The choice is made when the call is issued, so a captured CUDA graph keeps the
        choice of its capture: capture the drafts together with the selection (as ``run`` does), so
        that the graph's first draft writes the pack on every replay.  ``last`` marks the round's last
        draft: it reads the pack and then drops it from L2 unwritten, so the next draft writes it
        again."""
        idx = self.idx.view(self.kv.batch, self.kv.h_kv, self.k_max)
        cnt = self.cnt.view(self.kv.batch, self.kv.h_kv)
        o = out if out is not None else self.out_d
        if self.pack is None:
            return B.ssd_draft_attn(self.kv, q_draft, idx, cnt, self.scale, out=o, lse=self.lse_d, workspace=self.ws,
                                    stream=stream)
        if not self._packed:
            mode = B.PACK_WRITE
        else:
            mode = B.PACK_READ_DISCARD if last else B.PACK_READ
        self._packed = not (self._packed and last)
        return B.ssd_draft_attn_packed(self.kv, q_draft, idx, cnt, self.scale, self.pack, mode, out=o, lse=self.lse_d,
                                       workspace=self.ws, stream=stream)

    def draft_oracle_topk(self, q_draft: torch.Tensor, k_per_req: torch.Tensor, out: Optional[torch.Tensor] = None,
                          stream=None) -> dict:
        """Draft with the "oracle top-k" pattern (SparseSpec §3.3, the reference the pages measure
        drafts against): the draft query selects by its own exact criticality instead of by the last
        verify's.  Three calls: a verify pass with the draft query as the single candidate (it sees
        the whole cache) gives that criticality and the dense output; Top-K selects K_b tokens per
        (request, KV head); the sparse draft attends them.  Buffers are allocated on first use.
        Returns the sparse draft's ``out`` / ``lse`` plus ``dense`` (the full-attention output) and
        the selection ``idx`` / ``cnt``."""
        kv = self.kv
        Bsz, hkv, d = kv.batch, kv.h_kv, kv.d
        if not hasattr(self, "_o_scores"):
            dev = kv.device
            self._o_dense = torch.empty((Bsz, 1, self.h_q, d), dtype=torch.float32, device=dev)
            self._o_lse = torch.empty((Bsz, 1, self.h_q), dtype=torch.float32, device=dev)
            self._o_scores = torch.zeros((Bsz, hkv, max(kv.max_seq_len, 1)), dtype=torch.float32, device=dev)
            self._o_idx = torch.empty((Bsz * hkv, self.k_max), dtype=torch.int32, device=dev)
            self._o_cnt = torch.empty((Bsz * hkv,), dtype=torch.int32, device=dev)
            self._o_out = torch.empty((Bsz, self.h_q, d), dtype=torch.float32, device=dev)
            self._o_lse_d = torch.empty((Bsz, self.h_q), dtype=torch.float32, device=dev)
        B.ssd_verify_attn(kv, q_draft.view(Bsz, 1, self.h_q, d), 1, self.scale, out=self._o_dense, lse=self._o_lse,
                          scores=self._o_scores, workspace=self.ws, stream=stream)
        B.ssd_select_topk(self._o_scores, kv.seq_lens, k_per_req, self.k_max, hkv, max_len=kv.max_seq_len,
                          idx=self._o_idx, cnt=self._o_cnt, stream=stream)
        o = out if out is not None else self._o_out
        B.ssd_draft_attn(kv, q_draft, self._o_idx.view(Bsz, hkv, self.k_max), self._o_cnt.view(Bsz, hkv), self.scale,
                         out=o, lse=self._o_lse_d, workspace=self.ws, stream=stream)
        return {"out": o, "lse": self._o_lse_d, "dense": self._o_dense.view(Bsz, self.h_q, d),
                "scores": self._o_scores, "idx": self._o_idx, "cnt": self._o_cnt}

    def run(self, q_verify: torch.Tensor, q_drafts: torch.Tensor, k_per_req: torch.Tensor,
            draft_outs: Optional[torch.Tensor] = None, stream=None, fused_select: bool = False):
        """verify -> select -> len(q_drafts) drafts.  draft_outs [k, B, h_q, d] keeps every draft's
        output (else each overwrites ``out_d``).  fused_select runs the selection inside the verify's
        criticality pass (one launch fewer, same results)."""
        if fused_select:
            self.verify_select(q_verify, k_per_req, stream)
        else:
            self.verify(q_verify, stream)
            self.select(k_per_req, stream)
        k = q_drafts.shape[0]
        for j in range(k):
            self.draft(q_drafts[j], out=None if draft_outs is None else draft_outs[j], stream=stream,
                       last=j == k - 1)
