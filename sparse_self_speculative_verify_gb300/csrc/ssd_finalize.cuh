// ssd_finalize.cuh -- the per-unit pieces of the verify's finalize (LSE merge of a unit's splits,
// split combine, criticality rematerialisation), shared by the finalize and fused-select kernels
// (ssd_verify.cu) and by the tail pass of the tensor-core verify (ssd_verify_tc.cu), so that every
// path computes the same values bit for bit.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: the verify caches logits and the log-sum-exp so that the attention scores
// can be rematerialised; crit[t] = sum over the rows r of the unit of e[r][t] *
// 2^(m_ref[r][t >> ref_shift] - LSE2_r), with e the cached fp16 values and m_ref their log2 reference
// per 2^ref_shift tokens (16, or 128 from the tensor-core verify).
#pragma once

#include "ssd_topk.cuh"
#include "ssd_verify_tile.cuh"

namespace ssd {

constexpr int kFinAhead = 5;  // side-value rows loaded per batch

__device__ __forceinline__ void fin_fma_row(const uint4 &raw, float c, float (&acc)[8]) {
  const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 pf = __half22float2(h2[k]);
    acc[2 * k] = fmaf(pf.x, c, acc[2 * k]);
    acc[2 * k + 1] = fmaf(pf.y, c, acc[2 * k + 1]);
  }
}

// LSE merge of one unit's split log-sum-exps, per row r < R: sLn[r] (natural log) and sL2[r]
// (log2) of the row's total.  Warp w of an NW-warp block takes rows w, w + NW, ...; lane j holds
// split j (a loop when ns > 32).  Every split value is loaded before the first reduction.  Split
// partials are read through L2 only (they may have been written by other blocks of the same grid).
template <int NW>
__device__ __forceinline__ void fin_lse_merge(const FinalizeArgs &f, int64_t pbase, int ns, float *sLn, float *sL2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int Q = (kMaxRows + NW - 1) / NW;
  float v[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int r = warp + NW * q;
    v[q] = (r < f.R && lane < ns) ? __ldcg(f.lse_parts + pbase + (int64_t)lane * f.R + r) : -INFINITY;
  }
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int r = warp + NW * q;
    if (r >= f.R) break;
    float M = v[q];
    for (int j = lane + 32; j < ns; j += 32) M = fmaxf(M, __ldcg(f.lse_parts + pbase + (int64_t)j * f.R + r));
    M = warp_max(M);
    float sum = 0.f;
    if (M != -INFINITY) {
      sum = lane < ns ? fast_exp2((v[q] - M) * kLog2e) : 0.f;
      for (int j = lane + 32; j < ns; j += 32) sum += fast_exp2((__ldcg(f.lse_parts + pbase + (int64_t)j * f.R + r) - M) * kLog2e);
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      const float ln = (M == -INFINITY) ? -INFINITY : M + __logf(sum);
      sLn[r] = ln;
      sL2[r] = ln * kLog2e;
    }
  }
}

// Split combine of one unit (request b, KV head g): rows r = r0, r0 + rstep, ... each get
// out = sum_j 2^((lse_j - LSE) log2 e) o_j over the splits and lse = LSE; thread q4 of the D / 4
// threads of a row takes one float4 of d.
__device__ __forceinline__ void fin_combine_rows(const FinalizeArgs &f, int64_t pbase, int ns, const float *sLn,
                                                 int b, int g, int r0, int rstep, int q4) {
  const int D = f.D;
  for (int r = r0; r < f.R; r += rstep) {
    const float ln = sLn[r];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ln != -INFINITY) {
      const float *lp = f.lse_parts + pbase + r;
      const float4 *op = reinterpret_cast<const float4 *>(f.o_parts + (pbase + r) * D) + q4;
      const int64_t ostep = (int64_t)f.R * D / 4;
#pragma unroll 4
      for (int j = 0; j < ns; ++j) {
        float w = fast_exp2((__ldcg(lp + (int64_t)j * f.R) - ln) * kLog2e);
        float4 o = __ldcg(op + j * ostep);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    const int i = r / f.G, hl = r % f.G;
    const int64_t row = ((int64_t)b * f.n_c + i) * f.h_q + g * f.G + hl;
    reinterpret_cast<float4 *>(f.out + row * D)[q4] = acc;
    if (q4 == 0 && f.lse) f.lse[row] = ln;
  }
}

// Drops unit u's split partials (ns splits x R rows of D floats from row pbase, read for the last time
// by this block's combine) from L2 without writing them back.  Threads tid < nt of the block, after a
// barrier that follows the block's last read of them; every row starts 128-byte aligned.
__device__ __forceinline__ void fin_discard_parts(const FinalizeArgs &f, int64_t pbase, int ns, int tid, int nt) {
  const char *base = reinterpret_cast<const char *>(f.o_parts + pbase * f.D);
  const int lines = ns * f.R * f.D * 4 / 128;
  for (int e = tid; e < lines; e += nt) discard_l2_line(base + (int64_t)e * 128);
}

// Splits of unit u's request of length L, as the verify pass cut them.
__device__ __forceinline__ int fin_splits(const FinalizeArgs &f, int u, int L) {
  return f.ucnt       ? block_splits(min(max(f.ucnt[u], 0), f.umax))
         : f.balanced ? tc_split_count(L, tc_tail_split(f.split_len[0], u / f.h_kv, f.split_len[1]))
                      : verify_splits(L, f.split_len ? *f.split_len : kSplitTokens);
}


// Criticality of unit u (request length L) for threads tid < NT: thread tid takes eight consecutive
// tokens t0 = 8 tid, 8 (tid + NT), ...; rows are read in batches of kFinAhead (every load of a batch
// in flight together) and summed in row order with one fused multiply-add each, exactly as the
// finalize's token blocks do.  Writes scores[u][t] for t < L and, when s_keys is not null, the
// order-preserving keys into s_keys[t].  sL2 holds the rows' log2 LSEs.
template <int NT>
__device__ __forceinline__ void fin_unit_scores(const FinalizeArgs &f, int u, int L, const float *sL2, uint32_t *s_keys,
                                                int tid) {
  const int64_t rbase = (int64_t)u * f.R;
  const int nref = ref_stride(f.Lpad, f.ref_shift);
  const __half *sp = f.side_p + rbase * f.Lpad;
  for (int t0 = tid * 8; t0 < L; t0 += NT * 8) {
    const int grp = t0 >> f.ref_shift;
    float crit[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) crit[k] = 0.f;
    for (int r0 = 0; r0 < f.R; r0 += kFinAhead) {
      uint4 raw[kFinAhead];
      float m[kFinAhead];
#pragma unroll
      for (int k = 0; k < kFinAhead; ++k) {
        const int r = r0 + k;
        raw[k] = r < f.R ? __ldcg(reinterpret_cast<const uint4 *>(sp + (int64_t)r * f.Lpad + t0)) : make_uint4(0, 0, 0, 0);
        m[k] = r < f.R ? __ldcg(f.side_m + (rbase + r) * nref + grp) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kFinAhead; ++k) {
        const int r = r0 + k;
        if (r < f.R) {
          const float l2 = sL2[r];
          fin_fma_row(raw[k], (l2 == -INFINITY) ? 0.f : fast_exp2(m[k] - l2), crit);
        }
      }
    }
    float *dst = f.scores + (int64_t)u * f.scores_stride + t0;
    if (t0 + 8 <= L && ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
      reinterpret_cast<float4 *>(dst)[0] = make_float4(crit[0], crit[1], crit[2], crit[3]);
      reinterpret_cast<float4 *>(dst)[1] = make_float4(crit[4], crit[5], crit[6], crit[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (t0 + k < L) dst[k] = crit[k];
    }
    if (s_keys) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (t0 + k < L) s_keys[t0 + k] = score_key(crit[k]);
    }
  }
}

// Stores the K and V rows of unit u's n selected tokens (f.sel_idx[u][0, n)) into the row pack, as
// the draft's pack reader takes them: the unit's chunk c holds selection slots [64 c, 64 c + 64) as a
// K tile then a V tile of 64 rows; row j of a tile sits at j * row bytes with its 16-byte chunk ch at
// (ch ^ (j % 8)) * 16.  Rows past n are not stored.  Threads tid < NT of the block call it, after a
// barrier that makes the selection visible; s_rows is shared scratch of kPackBatch int64 entries.
// First each selected token's K-row byte offset in the pool is resolved once (page lookup; -1 for a
// page out of range, whose rows are stored as zeros: the verify has flagged SSD_FAULT_PAGE), then the
// rows are copied 16 bytes at a time, eight copies in flight per thread.
constexpr int kPackBatch = 1024;
template <int NT>
__device__ __forceinline__ void pack_unit_rows(const FinalizeArgs &f, int u, int n, int tid, int64_t *s_rows) {
  const int b = u / f.h_kv, g = u % f.h_kv;
  const int rowb = f.D * f.esize, cpr = rowb / 16;
  const int64_t tile = (int64_t)kDraftChunk * rowb;
  char *pu = f.pack + (int64_t)u * f.pack_cmax * 2 * tile;
  const int32_t *sel = f.sel_idx + (int64_t)u * f.sel_kmax;
  const char *pool = static_cast<const char *>(f.kv.pool);
  const int64_t v_off = (int64_t)f.kv.h_kv * f.kv.page_size * rowb;  // a page's K rows to its V rows
  for (int j0 = 0; j0 < n; j0 += kPackBatch) {
    const int nb = min(kPackBatch, n - j0);
    for (int j = tid; j < nb; j += NT) {
      const int t = sel[j0 + j];
      int64_t off = -1;
      if (t >= 0) {
        const int32_t p = __ldg(f.kv.page_table + (int64_t)b * f.kv.max_pages + (t >> f.kv.log2_ps));
        if (p >= 0 && (int64_t)p < f.kv.num_pages)
          off = ((((int64_t)p * 2) * f.kv.h_kv + g) * f.kv.page_size + (t & (f.kv.page_size - 1))) * rowb;
      }
      s_rows[j] = off;
    }
    __syncthreads();
    const int total = nb * 2 * cpr;
    constexpr int U = 8;
    for (int e0 = tid; e0 < total; e0 += NT * U) {
      uint4 v[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int e = e0 + k * NT;
        v[k] = make_uint4(0, 0, 0, 0);
        if (e < total) {
          const int j = e / (2 * cpr), kv = (e / cpr) & 1, ch = e % cpr;
          const int64_t off = s_rows[j];
          if (off >= 0) v[k] = __ldg(reinterpret_cast<const uint4 *>(pool + off + kv * v_off) + ch);
        }
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int e = e0 + k * NT;
        if (e < total) {
          const int j = e / (2 * cpr), kv = (e / cpr) & 1, ch = e % cpr;
          const int js = j0 + j, jr = js % kDraftChunk;
          *reinterpret_cast<uint4 *>(pu + ((int64_t)(js / kDraftChunk) * 2 + kv) * tile + (int64_t)jr * rowb +
                                     ((ch ^ (jr & 7)) << 4)) = v[k];
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace ssd
