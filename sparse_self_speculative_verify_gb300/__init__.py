"""GB300 (sm_103a) attention hot path of sparse self-speculative decoding.

Verify attention with fused criticality, Top-K selection, sparse draft attention, the unified
verify/draft launch and the block-granular variant, as CUDA kernels behind the C ABI in
``include/ssd.h``.  ``binding`` is the thin Python layer over that ABI; ``round`` strings the calls
of one speculative round together; ``workloads`` draws the seeded synthetic inputs.
"""

from .binding import (KVCache, LibraryNotBuilt, SSDError, Workspace, ssd_block_sparse_attn, ssd_block_union,
                      ssd_combine, ssd_draft_attn, ssd_draft_attn_packed, ssd_draft_attn_static,
                      ssd_draft_pack_bytes, ssd_kv_advance, ssd_kv_append,
                      ssd_phase_assign, ssd_phase_fill, ssd_select_topk, ssd_select_topp, ssd_status, ssd_unified_attn,
                      ssd_verify_attn, ssd_verify_select, ssd_version)
from .round import SpecRound

__all__ = ["KVCache", "LibraryNotBuilt", "SSDError", "Workspace", "SpecRound", "ssd_block_sparse_attn",
           "ssd_block_union", "ssd_combine", "ssd_draft_attn", "ssd_draft_attn_packed", "ssd_draft_attn_static",
           "ssd_draft_pack_bytes", "ssd_kv_advance",
           "ssd_kv_append", "ssd_phase_assign", "ssd_phase_fill", "ssd_select_topk", "ssd_select_topp",
           "ssd_status", "ssd_unified_attn", "ssd_verify_attn", "ssd_verify_select", "ssd_version"]
