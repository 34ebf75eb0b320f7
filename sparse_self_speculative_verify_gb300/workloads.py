"""Seeded synthetic workloads for sparse self-speculative decoding attention.

This module only draws random inputs and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle read the bytes it
produces, so it is the one module the two sides share.

Shapes follow the decode workloads the SparseSpec paper studies
("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding
with Sparse Attention": §3.1 / A1 Qwen3-8B at batch 128 and 8192 output tokens,
Table 1 output lengths, §5.4 sparsity s = 0.05) and the SpecSA post's block
selection ("SpecSA", overlap-aware grouped query execution).  The datasets and
model weights of those pages are not available, so the planted-direction
distribution below stands in for them:

* per (request, KV head) a unit direction u = g / |g|, g ~ N(0, I_d);
* Q = N(0, 1) + 2u for every query head of the group (candidates and drafts);
* K = N(0, 1), with round(0.02 * L) positions (uniform, without replacement)
  shifted by +4u;
* V = N(0, 1).

Values are rounded once to the storage dtype (bf16 or fp32).  The KV cache is
paged: pool[num_pages, 2, H_kv, page_size, d] (K at index 0, V at index 1), a
page table [B, max_pages] of int32 page ids (-1 where unused) and seq_lens [B].
Slots past a request's length inside its last page hold NaN, so a kernel that
reads them without masking fails parity instead of passing by luck.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

# --------------------------------------------------------------------------
# Workload descriptions (sizes only).
# --------------------------------------------------------------------------


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    batch: int
    h_q: int
    h_kv: int
    d: int
    dtype: str  # "bf16" or "f32"
    page_size: int
    k: int  # draft length; n_cand = k + 1 verify positions
    len_kind: str  # "fixed", "uniform", "lognormal"
    len_lo: int
    len_hi: int
    len_median: float = 0.0
    len_sigma: float = 0.0
    shuffled: bool = True
    topk_fixed: Optional[int] = None  # fixed top-K per (request, KV head)
    topk_frac: float = 0.05  # else ceil(frac * L)
    unified: bool = False  # requests mixed between verify and draft phases
    verify_prob: float = 0.0
    block_size: int = 0  # >0: block-granular selection
    top_blocks: int = 0

    @property
    def n_cand(self) -> int:
        return self.k + 1

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


SPECS = {
    # 2 requests x 512 tokens, 8/2 heads, d=64, fp32, one contiguous page per request.
    "tiny": WorkloadSpec("tiny", 2, 8, 2, 64, "f32", 512, 4, "fixed", 512, 512,
                         shuffled=False, topk_fixed=64),
    # Qwen3-8B attention layer: 32 requests, L ~ U[2048, 8192], 32/8 heads, d=128, bf16, page 16.
    "qwen3_8b": WorkloadSpec("qwen3_8b", 32, 32, 8, 128, "bf16", 16, 4, "uniform", 2048, 8192),
    # 128 requests x 8192, k = 6.
    "b128_l8k": WorkloadSpec("b128_l8k", 128, 32, 8, 128, "bf16", 16, 6, "fixed", 8192, 8192),
    # Qwen3-14B unified batch: 64 requests, lognormal lengths (median 13.5K, sigma 0.5), 40/8 heads.
    "qwen3_14b_unified": WorkloadSpec("qwen3_14b_unified", 64, 40, 8, 128, "bf16", 16, 4,
                                      "lognormal", 4096, 32768, len_median=13500.0,
                                      len_sigma=0.5, unified=True, verify_prob=0.2),
    # 8 requests x 131072, block-granular (64-token blocks, top-16 per candidate).
    "block_131k": WorkloadSpec("block_131k", 8, 32, 8, 128, "bf16", 16, 4, "fixed", 131072,
                               131072, block_size=64, top_blocks=16),
}

SPEC_ORDER = ["tiny", "qwen3_8b", "b128_l8k", "qwen3_14b_unified", "block_131k"]


def spec_seed(name: str) -> int:
    """Default seed: 1000 + the workload's position in SPEC_ORDER (1-based)."""
    return 1000 + SPEC_ORDER.index(name) + 1


def scaled_spec(spec: WorkloadSpec, **over) -> WorkloadSpec:
    """A copy of ``spec`` with some fields replaced (used for small test cases)."""
    d = dict(spec.__dict__)
    d.update(over)
    return WorkloadSpec(**d)


# --------------------------------------------------------------------------
# Generated workload.
# --------------------------------------------------------------------------


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    seq_lens: torch.Tensor  # [B] int32
    page_table: torch.Tensor  # [B, max_pages] int32, -1 unused
    pool: torch.Tensor  # [num_pages, 2, H_kv, page_size, d]
    q_verify: torch.Tensor  # [B, n_cand, H_q, d]
    q_draft: torch.Tensor  # [k, B, H_q, d] (one query per draft step)
    k_per_req: torch.Tensor  # [B] int32 top-K per (request, KV head)
    phase: Optional[torch.Tensor] = None  # [B] uint8: 1 = verify, 0 = draft
    extra: dict = field(default_factory=dict)

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item())

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def num_pages(self) -> int:
        return int(self.pool.shape[0])

    def kv_tokens(self) -> int:
        """Sum over requests of L_b (tokens, per KV head)."""
        return int(self.seq_lens.to(torch.int64).sum().item())


def _lengths(spec: WorkloadSpec, gen: torch.Generator) -> torch.Tensor:
    b = spec.batch
    if spec.len_kind == "fixed":
        return torch.full((b,), spec.len_lo, dtype=torch.int64)
    if spec.len_kind == "uniform":
        return torch.randint(spec.len_lo, spec.len_hi + 1, (b,), generator=gen, dtype=torch.int64)
    if spec.len_kind == "lognormal":
        z = torch.randn((b,), generator=gen, dtype=torch.float64)
        lens = torch.exp(math.log(spec.len_median) + spec.len_sigma * z)
        return torch.clamp(torch.round(lens), spec.len_lo, spec.len_hi).to(torch.int64)
    raise ValueError(spec.len_kind)


def top_k_for_length(spec: WorkloadSpec, length: int) -> int:
    """Top-K per (request, KV head): a fixed count, else ceil(s * L) with s = 0.05."""
    if spec.topk_fixed is not None:
        return min(spec.topk_fixed, length)
    return min(length, int(math.ceil(spec.topk_frac * length - 1e-9)))


def make_workload(spec: WorkloadSpec, seed: Optional[int] = None, device: str = "cpu",
                  lengths: Optional[list] = None, pad_value: float = float("nan"),
                  spare_pages: int = 0) -> Workload:
    """Draw one seeded workload of ``spec``'s shape on ``device``.

    ``lengths`` overrides the drawn sequence lengths (used by edge-case tests).
    The same (spec, seed, device type) always gives the same bytes.
    """
    if seed is None:
        seed = spec_seed(spec.name) if spec.name in SPECS else 1
    dev = torch.device(device)
    gen_cpu = torch.Generator(device="cpu").manual_seed(seed)
    gen = gen_cpu if dev.type == "cpu" else torch.Generator(device=dev).manual_seed(seed)

    B, Hq, Hkv, d, ps = spec.batch, spec.h_q, spec.h_kv, spec.d, spec.page_size
    G, nc = spec.group, spec.n_cand
    assert Hq % Hkv == 0
    lens = torch.tensor(lengths, dtype=torch.int64) if lengths is not None else _lengths(spec, gen_cpu)
    assert lens.numel() == B
    npages = [(int(L) + ps - 1) // ps for L in lens.tolist()]
    max_pages = max(1, max(npages))
    total_pages = sum(npages) + spare_pages
    perm = torch.randperm(total_pages, generator=gen_cpu) if spec.shuffled else torch.arange(total_pages)
    page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        page_table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n

    tdt = spec.torch_dtype
    pool = torch.full((total_pages, 2, Hkv, ps, d), pad_value, dtype=tdt, device=dev)
    u = torch.randn((B, Hkv, d), generator=gen, device=dev, dtype=torch.float32)
    u = u / u.norm(dim=-1, keepdim=True)
    pt_dev = page_table.to(dev)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        n = npages[b]
        k_b = torch.randn((Hkv, L, d), generator=gen, device=dev, dtype=torch.float32)
        v_b = torch.randn((Hkv, L, d), generator=gen, device=dev, dtype=torch.float32)
        n_plant = int(round(0.02 * L))
        if n_plant > 0:
            keys = torch.rand((Hkv, L), generator=gen, device=dev, dtype=torch.float32)
            pos = torch.topk(keys, n_plant, dim=1, largest=False).indices  # [Hkv, n_plant]
            rows = torch.arange(Hkv, device=dev).unsqueeze(1)
            k_b[rows, pos] += 4.0 * u[b].unsqueeze(1)
        padded = n * ps
        kk = torch.full((Hkv, padded, d), pad_value, device=dev, dtype=torch.float32)
        vv = torch.full((Hkv, padded, d), pad_value, device=dev, dtype=torch.float32)
        kk[:, :L] = k_b
        vv[:, :L] = v_b
        pages = pt_dev[b, :n].to(torch.int64)
        pool[pages, 0] = kk.view(Hkv, n, ps, d).permute(1, 0, 2, 3).to(tdt)
        pool[pages, 1] = vv.view(Hkv, n, ps, d).permute(1, 0, 2, 3).to(tdt)

    # Query heads h of KV group g = h // G share u[b, g].
    u_h = u.repeat_interleave(G, dim=1)  # [B, Hq, d]
    qv = torch.randn((B, nc, Hq, d), generator=gen, device=dev, dtype=torch.float32)
    qv = (qv + 2.0 * u_h.unsqueeze(1)).to(tdt)
    qd = torch.randn((max(spec.k, 1), B, Hq, d), generator=gen, device=dev, dtype=torch.float32)
    qd = (qd + 2.0 * u_h.unsqueeze(0)).to(tdt)

    kpr = torch.tensor([top_k_for_length(spec, int(L)) for L in lens.tolist()], dtype=torch.int32)
    phase = None
    if spec.unified:
        r = torch.rand((B,), generator=gen_cpu)
        phase = (r < spec.verify_prob).to(torch.uint8)
        if int(phase.sum()) == 0:
            phase[0] = 1
    return Workload(spec=spec, seed=seed, seq_lens=lens.to(torch.int32).to(dev),
                    page_table=pt_dev, pool=pool, q_verify=qv, q_draft=qd,
                    k_per_req=kpr.to(dev), phase=None if phase is None else phase.to(dev))


def random_index_sets(seq_lens: torch.Tensor, h_kv: int, k_per_req: torch.Tensor, k_max: int,
                      seed: int) -> tuple:
    """Sorted, distinct random token indices per (request, KV head): idx [B, H_kv, k_max]
    (-1 padded) and cnt [B, H_kv].  Used as draft inputs that do not come from any
    selection step."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    lens = seq_lens.cpu().tolist()
    ks = k_per_req.cpu().tolist()
    B = len(lens)
    idx = torch.full((B, h_kv, k_max), -1, dtype=torch.int32)
    cnt = torch.zeros((B, h_kv), dtype=torch.int32)
    for b in range(B):
        for g in range(h_kv):
            k = min(ks[b], lens[b], k_max)
            if k == 0:
                continue
            sel = torch.randperm(lens[b], generator=gen)[:k].sort().values
            idx[b, g, :k] = sel.to(torch.int32)
            cnt[b, g] = k
    return idx, cnt


def random_scores(n_rows: int, length: int, seed: int, ties: bool = True) -> torch.Tensor:
    """Non-negative fp32 score rows for selection tests; with ``ties`` many values repeat
    exactly (few distinct levels plus exact zeros)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.rand((n_rows, length), generator=gen, dtype=torch.float32)
    if ties:
        levels = torch.randint(0, 7, (n_rows, length), generator=gen).to(torch.float32) / 8.0
        pick = torch.rand((n_rows, length), generator=gen) < 0.5
        x = torch.where(pick, levels, x)
        zero = torch.rand((n_rows, length), generator=gen) < 0.1
        x = torch.where(zero, torch.zeros_like(x), x)
    return x.contiguous()


def flush_buffer(device, nbytes: int = 512 << 20) -> torch.Tensor:
    """A scratch buffer larger than L2, written between timed iterations when requested."""
    return torch.empty(nbytes // 4, dtype=torch.float32, device=device)
