// ssd_draft_tile.cuh -- one draft work item: up to kDraftChunk selected tokens of one (request b,
// KV head g), all G query heads of the group.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: the k drafts after a verify load and attend only the critical tokens the
// verify selected; §4.2: sparse attention is PagedAttention with page size 1, i.e. attention over an
// explicit token list.  The selected K and V rows are gathered into swizzled shared memory with
// 16-byte cp.async (one K row = one contiguous 256-byte line of the page).  The two contractions
// are small (G query rows against 64 tokens) but still dominate the instruction count, so for bf16
// caches they run on tensor cores (mma.sync m16n8k16: S^T = K Q^T with the queries as register B
// fragments, O^T = V^T P^T with P as bf16 high + residual parts); fp32 caches use CUDA cores.  The
// chunk's partial result is merged with the other chunks of the same (request, KV head) by the last
// chunk to finish (atomic ticket, no wait).
//
// All k drafts of a round attend the same selected set (SparseSpec §4.1: the pattern is refreshed
// only by the next verify), so the first draft can store each chunk's gathered K and V tiles, as
// they sit in shared memory, into a contiguous "row pack" (bf16: one bulk store per tile); the later
// drafts copy those tiles back and skip the index, length and page-table lookups and the scattered
// 256-byte row reads (bf16: draft_pack_unit below, one bulk copy per tile on an mbarrier, one block
// per (request, KV head); fp32: this chunk kernel with linear cp.async).  Pack layout: [unit][chunk]
// [K tile, V tile], each tile kDraftChunk rows of D elements in the swizzled shared-memory order;
// rows past the chunk's count are neither stored nor read.
#pragma once

#include "ssd_common.cuh"
#include "ssd_sm100.cuh"

namespace ssd {

// 1-D bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from this block's
// shared memory to global, in the thread's bulk group.  The shared source may be overwritten once
// bulk_wait_read() has returned.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Bounded wait of a thread for a bulk tile load (about a second at the SM clock); on expiry the
// status word gets SSD_FAULT_TIMEOUT and the wait reports false.
constexpr long long kDraftWaitCycles = 2000000000ll;
__device__ __forceinline__ bool draft_tile_wait(uint32_t bar, uint32_t parity, unsigned *status) {
  if (sm100::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!sm100::mbar_try_wait_sleep(bar, parity, 20000u))
    if (clock64() - t0 > kDraftWaitCycles) {
      atomicOr(status, (unsigned)SSD_FAULT_TIMEOUT);
      return false;
    }
  return true;
}

struct DraftArgs {
  KVView kv;
  const void *q;  // [B][h_q][D]
  int h_q, G, k_max;
  const int32_t *idx;  // [B][h_kv][k_max]
  const int32_t *cnt;  // [B][h_kv]
  float scale_log2;
  int C_max;           // chunks per unit in the partial arrays
  float *o_parts;      // [units][C_max][G][D]
  float *lse_parts;    // [units][C_max][G]
  unsigned *counters;  // [units], zero between calls
  float *out;          // [B][h_q][D]
  float *lse;          // [B][h_q] or nullptr
  const uint8_t *phase;  // unified launch: draft items only for phase == 0 (nullptr otherwise)
  int defer_wait;        // unified launch: see draft_kernel
  char *pack;            // row pack [units][C_max][2][TILE] (pack_mode != SSD_PACK_NONE)
  int pack_mode;         // SSD_PACK_NONE / SSD_PACK_WRITE (gather, then store the tiles) / SSD_PACK_READ
  int pack_discard;      // SSD_PACK_READ_DISCARD: the pack reader drops the unit's pack lines from L2
  unsigned *status;
};

template <int D, typename T, int GMAX>
struct DraftCfg {
  static constexpr int ROWB = D * (int)sizeof(T);  // bytes of one K or V row
  static constexpr int CPR = ROWB / 16;
  static constexpr int TILE = kDraftChunk * ROWB;
  // bf16 (tensor-core path): one row tile, K then V, so that twice as many blocks fit on an SM;
  // fp32: a K tile and a V tile.  Then the queries (fp32; the output rows on the tensor-core path),
  // logits, row max / sum, row offsets, and (tensor-core path) P as bf16 high + residual parts.
  static constexpr bool TC = sizeof(T) == 2;
  static constexpr int SMEM = (TC ? 1 : 2) * TILE + (GMAX * D + GMAX * kDraftChunk + 2 * GMAX) * 4 +
                              kDraftChunk * 8 + (TC ? 2 * GMAX * kDraftChunk * 2 : 0);
};

__device__ __forceinline__ int draft_chunks(int n) { return n <= 0 ? 1 : cdiv(n, kDraftChunk); }

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &v, float *f);
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &v, float *f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &v, float *f) {
  f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

// ---- Tensor-core pieces of a bf16 draft chunk (mma.sync m16n8k16, fp32 accumulate) -------------
// The queries stay in registers as B fragments; K and V come from a swizzled row tile in shared
// memory through ldmatrix; P goes through bf16 high + residual parts (about 16 bits).
template <int D, int GMAX>
struct DraftMma {
  static constexpr int NT8 = (GMAX + 7) / 8;  // 8-wide head tiles
  static constexpr int KS = D / 16;           // 16-wide steps over d
  static constexpr int MTW = D / 16 / 4;      // 16-row d tiles per warp (4 warps) in P V
  static constexpr int ROWB = D * 2;
};

// B fragments of Q^T for query heads g G .. g G + G - 1 of request b: head n = 8 nt + lane / 4,
// dims k0, k0 + 1 and k0 + 8, k0 + 9 (zero for heads past G).
template <int D, int GMAX>
__device__ __forceinline__ void draft_q_frags(const void *q, int64_t row0, int G, int lane,
                                              uint32_t (&qb)[DraftMma<D, GMAX>::NT8][DraftMma<D, GMAX>::KS][2]) {
  using M = DraftMma<D, GMAX>;
  const unsigned short *q16 = reinterpret_cast<const unsigned short *>(q);
#pragma unroll
  for (int nt = 0; nt < M::NT8; ++nt) {
    const int hn = nt * 8 + (lane >> 2);
    const unsigned short *qr = q16 + (row0 + (hn < G ? hn : 0)) * D + (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < M::KS; ++ks) {
      uint32_t v0 = 0, v1 = 0;
      if (hn < G) {
        v0 = (uint32_t)__ldg(qr + ks * 16) | ((uint32_t)__ldg(qr + ks * 16 + 1) << 16);
        v1 = (uint32_t)__ldg(qr + ks * 16 + 8) | ((uint32_t)__ldg(qr + ks * 16 + 9) << 16);
      }
      qb[nt][ks][0] = v0;
      qb[nt][ks][1] = v1;
    }
  }
}

// Logits S^T = K Q^T of the chunk into sS[h][j] (scaled to log2 units; -inf for j >= n): warp w
// takes tokens 16w .. 16w + 15, its A fragments by ldmatrix from the swizzled K tile (thread t
// addresses row (t & 7) + 8 ((t >> 3) & 1), 16-byte chunk 2 ks + (t >> 4)).
template <int D, int GMAX>
__device__ __forceinline__ void draft_logits_mma(const char *sKt,
                                                 const uint32_t (&qb)[DraftMma<D, GMAX>::NT8][DraftMma<D, GMAX>::KS][2],
                                                 float *sS, int n, float scale_log2, int G, int warp, int lane) {
  using M = DraftMma<D, GMAX>;
  float acc[M::NT8][4];
#pragma unroll
  for (int nt = 0; nt < M::NT8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const int ar = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int ks = 0; ks < M::KS; ++ks) {
    const int ch = 2 * ks + (lane >> 4);
    uint32_t af[4];
    ldsm_x4(smem_u32(sKt + ar * M::ROWB + swz_chunk(ar, ch) * 16), af[0], af[1], af[2], af[3]);
#pragma unroll
    for (int nt = 0; nt < M::NT8; ++nt) mma_bf16(acc[nt], af, qb[nt][ks][0], qb[nt][ks][1]);
  }
  // c0, c1: token 16w + lane / 4, heads 8 nt + 2 (lane & 3) + {0, 1}; c2, c3: token + 8.
#pragma unroll
  for (int nt = 0; nt < M::NT8; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = warp * 16 + (lane >> 2) + (e >> 1) * 8, h = nt * 8 + (lane & 3) * 2 + (e & 1);
      if (h < G) sS[h * kDraftChunk + j] = (j < n) ? acc[nt][e] * scale_log2 : -INFINITY;
    }
  }
}

// Writes head h's probabilities p0 (token lane) and p1 (token lane + 32) as bf16 high + residual
// parts into sP [2][GMAX][chunk].
template <int GMAX>
__device__ __forceinline__ void draft_store_p(uint16_t *sP, int h, int lane, float p0, float p1) {
  uint32_t hi, lo;
  split_bf16(p0, p1, hi, lo);
  sP[h * kDraftChunk + lane] = (uint16_t)(hi & 0xffffu);
  sP[h * kDraftChunk + lane + 32] = (uint16_t)(hi >> 16);
  sP[(GMAX + h) * kDraftChunk + lane] = (uint16_t)(lo & 0xffffu);
  sP[(GMAX + h) * kDraftChunk + lane + 32] = (uint16_t)(lo >> 16);
}

// o += V^T P^T over the chunk: warp w takes d rows 16 mt .. 16 mt + 15 for mt = w MTW ..; A
// fragments by transposing ldmatrix from the swizzled V tile, B fragments (P^T) from the bf16 P
// parts.  Accumulator element e of o[mi][nt] sits at d = 16 mt + lane / 4 (+ 8 for e >= 2), head
// 8 nt + 2 (lane & 3) + (e & 1).
template <int D, int GMAX>
__device__ __forceinline__ void draft_pv_mma(const char *sVt, const uint16_t *sP, int G, int warp, int lane,
                                             float (&o)[DraftMma<D, GMAX>::MTW][DraftMma<D, GMAX>::NT8][4]) {
  using M = DraftMma<D, GMAX>;
#pragma unroll
  for (int ks = 0; ks < kDraftChunk / 16; ++ks) {
    uint32_t bh[M::NT8][2], bl[M::NT8][2];
#pragma unroll
    for (int nt = 0; nt < M::NT8; ++nt) {
      const int hn = nt * 8 + (lane >> 2), k0 = ks * 16 + (lane & 3) * 2;
      bh[nt][0] = bh[nt][1] = bl[nt][0] = bl[nt][1] = 0u;
      if (hn < G) {
        bh[nt][0] = *reinterpret_cast<const uint32_t *>(sP + hn * kDraftChunk + k0);
        bh[nt][1] = *reinterpret_cast<const uint32_t *>(sP + hn * kDraftChunk + k0 + 8);
        bl[nt][0] = *reinterpret_cast<const uint32_t *>(sP + (GMAX + hn) * kDraftChunk + k0);
        bl[nt][1] = *reinterpret_cast<const uint32_t *>(sP + (GMAX + hn) * kDraftChunk + k0 + 8);
      }
    }
    const int tr = ks * 16 + (lane & 7) + ((lane >> 4) << 3);  // token row of this thread's address
#pragma unroll
    for (int mi = 0; mi < M::MTW; ++mi) {
      const int ch = 2 * (warp * M::MTW + mi) + ((lane >> 3) & 1);
      uint32_t af[4];
      ldsm_x4_t(smem_u32(sVt + tr * M::ROWB + swz_chunk(tr, ch) * 16), af[0], af[1], af[2], af[3]);
#pragma unroll
      for (int nt = 0; nt < M::NT8; ++nt) {
        mma_bf16(o[mi][nt], af, bh[nt][0], bh[nt][1]);
        mma_bf16(o[mi][nt], af, bl[nt][0], bl[nt][1]);
      }
    }
  }
}

template <int D, typename T, int GMAX>
__device__ __forceinline__ void draft_item(const DraftArgs &a, int unit, int chunk, char *smem) {
  using C = DraftCfg<D, T, GMAX>;
  constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h_kv = a.kv.h_kv;
  const int b = unit / h_kv, g = unit % h_kv, G = a.G;
  // The list length, the request length and this chunk's token indices are loaded together (none
  // depends on another), so a block waits for one memory latency before it can resolve its rows.
  const bool from_pack = a.pack_mode == SSD_PACK_READ, to_pack = a.pack_mode == SSD_PACK_WRITE;
  const int j0 = chunk * kDraftChunk;
  int t_mine = -1;
  if (!from_pack && tid < kDraftChunk && j0 + tid < a.k_max) t_mine = __ldg(a.idx + (int64_t)unit * a.k_max + j0 + tid);
  const int L = from_pack ? 0 : effective_len(a.kv, b, 0, a.status);
  int n_all = a.cnt[unit];
  if (n_all < 0 || n_all > a.k_max) {
    atomicOr(a.status, (unsigned)SSD_FAULT_KMAX);
    n_all = n_all < 0 ? 0 : a.k_max;
  }
  const int n_chunks = draft_chunks(n_all);
  if (chunk >= n_chunks) return;
  const int n = min(kDraftChunk, n_all - j0);  // may be 0 for an empty list
  constexpr bool TC = C::TC;

  char *sKt = smem;
  char *sVt = TC ? smem : smem + C::TILE;  // the tensor-core path loads V into the K tile after the logits
  float *sQ = reinterpret_cast<float *>(smem + (TC ? 1 : 2) * C::TILE);  // [GMAX][D]
  float *sS = sQ + GMAX * D;                                   // [GMAX][kDraftChunk]
  float *sM = sS + GMAX * kDraftChunk;                         // [GMAX]
  float *sL = sM + GMAX;                                       // [GMAX]
  int64_t *sRow = reinterpret_cast<int64_t *>(sL + GMAX);       // [kDraftChunk] K row element offset, -1: none

  // This chunk's K and V tiles in the row pack.
  char *pk = a.pack ? a.pack + ((int64_t)unit * a.C_max + chunk) * (2 * C::TILE) : nullptr;
  // Copies a landed tile's first n rows to the pack (16-byte words in shared-memory order).
  auto store_tile = [&](char *dst, const char *src) {
    for (int c = tid; c < n * C::CPR; c += blockDim.x)
      reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
  };

  // Each token's K row, resolved once by its own thread (index check, page-table lookup).
  if (!from_pack && tid < kDraftChunk) {
    int64_t row = -1;
    if (tid < n) {
      if (t_mine >= 0 && t_mine < L) {
        const int32_t p = __ldg(a.kv.page_table + (int64_t)b * a.kv.max_pages + (t_mine >> a.kv.log2_ps));
        if (p >= 0 && (int64_t)p < a.kv.num_pages)
          row = ((((int64_t)p * 2) * h_kv + g) * a.kv.page_size + (t_mine & (a.kv.page_size - 1))) * D;
        else
          atomicOr(a.status, (unsigned)SSD_FAULT_PAGE);
      } else {
        atomicOr(a.status, (unsigned)SSD_FAULT_INDEX);
      }
    }
    sRow[tid] = row;
  }
  __syncthreads();

  // Gather the chunk's K and V rows (rows of skipped tokens are zero-filled), or copy the packed tiles
  // (rows past n zero-filled).  bf16 reads of the pack normally run draft_pack_unit instead.
  const int64_t v_off = (int64_t)h_kv * a.kv.page_size * D;
  if (from_pack) {
    for (int c = tid; c < kDraftChunk * C::CPR; c += blockDim.x) {
      const int sz = c / C::CPR < n ? 16 : 0;
      cp_async16(smem_u32(sKt + c * 16), pk + c * 16, sz);
      if (!TC) cp_async16(smem_u32(sVt + c * 16), pk + C::TILE + c * 16, sz);
    }
  } else
  for (int c = tid; c < kDraftChunk * C::CPR; c += blockDim.x) {
    int j = c / C::CPR, ch = c % C::CPR;
    const int64_t row = sRow[j];
    const T *kr = row >= 0 ? reinterpret_cast<const T *>(a.kv.pool) + row : nullptr;
    uint32_t off = j * C::ROWB + swz_chunk(j, ch) * 16;
    cp_async16(smem_u32(sKt + off), kr ? (const void *)(kr + ch * EPC) : a.kv.pool, kr ? 16 : 0);
    if (!TC) cp_async16(smem_u32(sVt + off), kr ? (const void *)(kr + v_off + ch * EPC) : a.kv.pool, kr ? 16 : 0);
  }
  cp_async_commit();
  // bf16 caches: logits and P V on tensor cores (DraftMma); fp32 caches: CUDA cores.
  using MM = DraftMma<D, GMAX>;
  const T *q = reinterpret_cast<const T *>(a.q);
  uint32_t qb[MM::NT8][MM::KS][2];
  if constexpr (TC) {
    draft_q_frags<D, GMAX>(a.q, (int64_t)b * a.h_q + g * G, G, lane, qb);
  } else {
    for (int e = tid; e < G * D; e += blockDim.x) {
      int hl = e / D, dd = e % D;
      sQ[e] = to_f32<T>(q[((int64_t)b * a.h_q + g * G + hl) * D + dd]);
    }
  }
  cp_async_wait<0>();
  // Every thread's landed rows are made visible to the bulk store (async proxy) before the barrier.
  if (TC && to_pack) sm100::fence_proxy_async_smem();
  __syncthreads();
  if (to_pack) {
    if constexpr (TC) {
      // One bulk store of the landed K rows; its reads of the tile finish before the V rows are
      // gathered into it.
      if (tid == 0 && n > 0) {
        bulk_store(pk, smem_u32(sKt), (uint32_t)(n * C::ROWB));
        bulk_commit();
      }
    } else {
      store_tile(pk, sKt);
      store_tile(pk + C::TILE, sVt);
    }
  }

  if constexpr (TC) {
    draft_logits_mma<D, GMAX>(sKt, qb, sS, n, a.scale_log2, G, warp, lane);
  } else {
    // Logits: thread pair (2j, 2j+1) computes token j, one half of d each.
    const int j = tid >> 1, half = tid & 1;
    float acc[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
#pragma unroll 4
    for (int c = 0; c < C::CPR / 2; ++c) {
      int ch = half * (C::CPR / 2) + c;
      uint4 raw = *reinterpret_cast<const uint4 *>(sKt + j * C::ROWB + swz_chunk(j, ch) * 16);
      float kf[EPC];
      unpack16<T>(raw, kf);
      const int d0 = ch * EPC;
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
          const float *qh = sQ + h * D + d0;
#pragma unroll
          for (int e = 0; e < EPC; ++e) acc[h] = fmaf(qh[e], kf[e], acc[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float s = acc[h] + __shfl_xor_sync(0xffffffffu, acc[h], 1);
      if (half == 0 && h < G) sS[h * kDraftChunk + j] = (j < n) ? s * a.scale_log2 : -INFINITY;
    }
  }
  if (TC && to_pack && tid == 0) bulk_wait_read();  // the K tile may be overwritten after the barrier
  __syncthreads();
  // P in bf16 high + residual parts [2][GMAX][kDraftChunk] for the tensor-core P V, after the row
  // offsets.
  uint16_t *sP = reinterpret_cast<uint16_t *>(sRow + kDraftChunk);
  if constexpr (TC) {
    // V rows into the tile the K rows occupied (every thread is past the logits and its pack
    // stores); they land while the softmax runs.
    if (from_pack) {
      for (int c = tid; c < kDraftChunk * C::CPR; c += blockDim.x)
        cp_async16(smem_u32(sVt + c * 16), pk + C::TILE + c * 16, c / C::CPR < n ? 16 : 0);
    } else
    for (int c = tid; c < kDraftChunk * C::CPR; c += blockDim.x) {
      const int j = c / C::CPR, ch = c % C::CPR;
      const int64_t row = sRow[j];
      const T *kr = row >= 0 ? reinterpret_cast<const T *>(a.kv.pool) + row : nullptr;
      cp_async16(smem_u32(sVt + j * C::ROWB + swz_chunk(j, ch) * 16), kr ? (const void *)(kr + v_off + ch * EPC)
                                                                            : a.kv.pool, kr ? 16 : 0);
    }
    cp_async_commit();
  }

  pdl_trigger();
  // Softmax over the chunk, one warp per head.
  for (int h = warp; h < G; h += blockDim.x / 32) {
    float v0 = sS[h * kDraftChunk + lane], v1 = sS[h * kDraftChunk + lane + 32];
    float m = warp_max(fmaxf(v0, v1));
    float base = (m == -INFINITY) ? 0.f : m;
    float p0 = fast_exp2(v0 - base), p1 = fast_exp2(v1 - base);
    sS[h * kDraftChunk + lane] = p0;
    sS[h * kDraftChunk + lane + 32] = p1;
    if constexpr (TC) draft_store_p<GMAX>(sP, h, lane, p0, p1);
    float l = warp_sum(p0 + p1);
    if (lane == 0) {
      sM[h] = m;
      sL[h] = l;
    }
  }
  __syncthreads();

  constexpr int NPAIR = D / 2;
  constexpr int PARTS = TC ? 1 : 128 / NPAIR;
  // [PARTS][GMAX][D]: the query area on the tensor-core path (the queries live in registers), the
  // K tile (free after the logits) on the CUDA-core path.
  float *red = TC ? sQ : reinterpret_cast<float *>(sKt);
  if constexpr (TC) {
    cp_async_wait<0>();
    if (to_pack) sm100::fence_proxy_async_smem();  // as for the K rows
    __syncthreads();
    if (to_pack && tid == 0 && n > 0) {
      bulk_store(pk + C::TILE, smem_u32(sVt), (uint32_t)(n * C::ROWB));
      bulk_commit();
    }
    float o[MM::MTW][MM::NT8][4];
#pragma unroll
    for (int mi = 0; mi < MM::MTW; ++mi)
#pragma unroll
      for (int nt = 0; nt < MM::NT8; ++nt) o[mi][nt][0] = o[mi][nt][1] = o[mi][nt][2] = o[mi][nt][3] = 0.f;
    draft_pv_mma<D, GMAX>(sVt, sP, G, warp, lane, o);
#pragma unroll
    for (int mi = 0; mi < MM::MTW; ++mi)
#pragma unroll
      for (int nt = 0; nt < MM::NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dd = (warp * MM::MTW + mi) * 16 + (lane >> 2) + (e >> 1) * 8;
          const int h = nt * 8 + (lane & 3) * 2 + (e & 1);
          if (h < G) red[h * D + dd] = o[mi][nt][e];
        }
    __syncthreads();
    if (to_pack && tid == 0) bulk_wait_read();  // the V tile's bulk store has read it
  } else {
  // O = P V: thread = (pair of d columns, token part).
  constexpr int TPP = kDraftChunk / PARTS;  // tokens per part
  const int dp = tid % NPAIR, part = tid / NPAIR;
  float acc0[GMAX], acc1[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) acc0[h] = acc1[h] = 0.f;
  {
    const int byte = dp * 2 * (int)sizeof(T);
    const int ch = byte / 16, within = byte % 16;
    for (int jj = 0; jj < TPP; ++jj) {
      int j = part * TPP + jj;
      const char *src = sVt + j * C::ROWB + swz_chunk(j, ch) * 16 + within;
      float v0, v1;
      if (sizeof(T) == 2) {
        uint32_t w = *reinterpret_cast<const uint32_t *>(src);
        v0 = bf16_lo(w);
        v1 = bf16_hi(w);
      } else {
        float2 w = *reinterpret_cast<const float2 *>(src);
        v0 = w.x;
        v1 = w.y;
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
          float p = sS[h * kDraftChunk + j];
          acc0[h] = fmaf(p, v0, acc0[h]);
          acc1[h] = fmaf(p, v1, acc1[h]);
        }
      }
    }
  }
  __syncthreads();  // K tile is free: reuse it for the part reduction
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    if (h < G) {
      red[(part * GMAX + h) * D + 2 * dp] = acc0[h];
      red[(part * GMAX + h) * D + 2 * dp + 1] = acc1[h];
    }
  }
  __syncthreads();
  }

  const bool single = (n_chunks == 1);
  const int64_t prow = ((int64_t)unit * a.C_max + chunk) * GMAX;
  for (int e = tid; e < G * D; e += blockDim.x) {
    int h = e / D, dd = e % D;
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < PARTS; ++p) s += red[(p * GMAX + h) * D + dd];
    float l = sL[h];
    bool empty = !(l > 0.f);
    float ov = empty ? 0.f : s / l;
    float lv = empty ? -INFINITY : (sM[h] + __log2f(l)) * kLn2;
    if (single) {
      int64_t row = (int64_t)b * a.h_q + g * G + h;
      a.out[row * D + dd] = ov;
      if (dd == 0 && a.lse) a.lse[row] = lv;
    } else {
      a.o_parts[(prow + h) * D + dd] = ov;
      if (dd == 0) a.lse_parts[prow + h] = lv;
    }
  }
  if (single) return;

  // Last chunk of this unit to finish merges all chunks (no waiting on other blocks).
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_last;
  if (tid == 0) s_last = (atomicAdd(a.counters + unit, 1u) == (unsigned)(n_chunks - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Per head: LSE over the chunks (one warp, lanes over chunks).
  const int64_t cbase = (int64_t)unit * a.C_max * GMAX;
  for (int h = warp; h < G; h += blockDim.x / 32) {
    float M = -INFINITY;
    for (int c = lane; c < n_chunks; c += 32) M = fmaxf(M, __ldcg(a.lse_parts + cbase + (int64_t)c * GMAX + h));
    M = warp_max(M);
    float s = 0.f;
    if (M != -INFINITY)
      for (int c = lane; c < n_chunks; c += 32)
        s += fast_exp2((__ldcg(a.lse_parts + cbase + (int64_t)c * GMAX + h) - M) * kLog2e);
    s = warp_sum(s);
    if (lane == 0) {
      sM[h] = M;
      sL[h] = s;
    }
  }
  __syncthreads();
  // Outputs: one float4 of d per thread, chunks unrolled (independent loads).
  for (int e = tid; e < G * (D / 4); e += blockDim.x) {
    const int h = e / (D / 4), q4 = e % (D / 4);
    const float M = sM[h], s = sL[h];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 4
      for (int c = 0; c < n_chunks; ++c) {
        const int64_t pr = cbase + (int64_t)c * GMAX + h;
        const float w = fast_exp2((__ldcg(a.lse_parts + pr) - M) * kLog2e);
        const float4 o = __ldcg(reinterpret_cast<const float4 *>(a.o_parts + pr * D) + q4);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    const bool ok = s > 0.f;
    const float inv = ok ? 1.f / s : 0.f;
    const int64_t row = (int64_t)b * a.h_q + g * G + h;
    reinterpret_cast<float4 *>(a.out + row * D)[q4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (q4 == 0 && a.lse) a.lse[row] = ok ? M + __logf(s) : -INFINITY;
  }
  if (tid == 0) a.counters[unit] = 0u;
}

// ---- Per-warp online softmax over a unit's chunks (bf16, tensor cores) ---------------------------
// One block of four warps per (request, KV head).  Each warp owns 16 rows of every chunk and runs its
// own online softmax over them: its logits stay in registers, its running max and sum per head and
// its P V accumulators are its own, and its probabilities go from the logits' accumulator layout to
// the P V operand layout by an 8x8 register transpose (movmatrix), so a chunk needs no exchange
// between warps.  The four warps' states are merged once at the end (LSE merge in a fixed order).

// 8x8 transpose of 16-bit elements held one 32-bit pair per thread in the mma fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t v) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}

// A warp's state.  Thread (lane) holds heads 8 nt + 2 (lane & 3) + {0, 1}: their running max and sum
// (log2 domain), and the P V accumulators o[mi][nt][e] at d = 16 mi + lane / 4 (+ 8 for e >= 2),
// head 8 nt + 2 (lane & 3) + (e & 1); qb holds the queries as B fragments.
template <int D, int GMAX>
struct DraftWarp {
  static constexpr int NT8 = DraftMma<D, GMAX>::NT8, KS = DraftMma<D, GMAX>::KS, MT = D / 16;
  static constexpr int GMAX8 = NT8 * 8;
  uint32_t qb[NT8][KS][2];
  float o[MT][NT8][4];
  float m_run[NT8][2], l_run[NT8][2];

  __device__ __forceinline__ void init(const DraftArgs &a, int b, int g, int lane) {
    draft_q_frags<D, GMAX>(a.q, (int64_t)b * a.h_q + g * a.G, a.G, lane, qb);
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) o[mi][nt][0] = o[mi][nt][1] = o[mi][nt][2] = o[mi][nt][3] = 0.f;
    }
  }

  // Rows r0 .. r0 + 15 of a chunk of n rows (swizzled K and V tiles; V rows at or past n must hold
  // finite values, their P is 0): logits, online softmax, P V.
  __device__ __forceinline__ void chunk(const char *sKt, const char *sVt, int n, int r0, float scale_log2, int lane) {
    using MM = DraftMma<D, GMAX>;
    float sacc[NT8][4];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    {
      // S^T = K Q^T (A fragments by ldmatrix from the swizzled K tile).
      const int ar = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int ch = 2 * ks + (lane >> 4);
        uint32_t af[4];
        ldsm_x4(smem_u32(sKt + ar * MM::ROWB + swz_chunk(ar, ch) * 16), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) mma_bf16(sacc[nt], af, qb[nt][ks][0], qb[nt][ks][1]);
      }
    }
    // Online softmax, per head: rows lane / 4 and lane / 4 + 8 are this thread's; the 8 lanes with
    // the same lane & 3 hold the warp's other rows of the same heads.
    const bool in0 = r0 + (lane >> 2) < n, in1 = r0 + (lane >> 2) + 8 < n;
    uint32_t pb_hi[NT8][2], pb_lo[NT8][2];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
      float p[4], alpha[2];
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const float v0 = in0 ? sacc[nt][e2] * scale_log2 : -INFINITY;
        const float v1 = in1 ? sacc[nt][2 + e2] * scale_log2 : -INFINITY;
        float mx = fmaxf(v0, v1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[nt][e2], mx);
        const float base = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[e2] = fast_exp2(m_run[nt][e2] - base);  // 0 before the first rows (m_run = -inf)
        p[e2] = fast_exp2(v0 - base);
        p[2 + e2] = fast_exp2(v1 - base);
        float ps = p[e2] + p[2 + e2];
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l_run[nt][e2] = l_run[nt][e2] * alpha[e2] + ps;
        m_run[nt][e2] = m_new;
      }
#pragma unroll
      for (int mi = 0; mi < MT; ++mi)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mi][nt][e] *= alpha[e & 1];
      // P as bf16 high part + residual, rows lane / 4 (pair 0) and + 8 (pair 1), heads in pairs;
      // transposed 8x8 blocks are the P^T operand: k = row 2 (lane & 3) + {0, 1}, n = head lane / 4.
      uint32_t h0, l0, h1, l1;
      split_bf16(p[0], p[1], h0, l0);
      split_bf16(p[2], p[3], h1, l1);
      pb_hi[nt][0] = movmatrix_t(h0);
      pb_hi[nt][1] = movmatrix_t(h1);
      pb_lo[nt][0] = movmatrix_t(l0);
      pb_lo[nt][1] = movmatrix_t(l1);
    }
    // O^T += V^T P^T over the warp's rows (A fragments by transposing ldmatrix from the V tile).
    const int tr = r0 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      const int ch = 2 * mi + ((lane >> 3) & 1);
      uint32_t af[4];
      ldsm_x4_t(smem_u32(sVt + tr * MM::ROWB + swz_chunk(tr, ch) * 16), af[0], af[1], af[2], af[3]);
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt) {
        mma_bf16(o[mi][nt], af, pb_hi[nt][0], pb_hi[nt][1]);
        mma_bf16(o[mi][nt], af, pb_lo[nt][0], pb_lo[nt][1]);
      }
    }
  }

  // Merges the four warps (fixed order: M = max_w m_w, L = sum_w 2^(m_w - M) l_w, O = sum_w
  // 2^(m_w - M) O_w) and writes the normalised output and LSE of request b's heads g G ..  Called by
  // the whole block after its last use of the scratch areas: sO [4][GMAX8][D] fp32, sWM and sWL
  // [4][GMAX8].
  __device__ __forceinline__ void merge_store(const DraftArgs &a, int b, int g, float *sO, float *sWM, float *sWL) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, G = a.G;
    if (lane < 4) {
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          sWM[warp * GMAX8 + nt * 8 + 2 * lane + e2] = m_run[nt][e2];
          sWL[warp * GMAX8 + nt * 8 + 2 * lane + e2] = l_run[nt][e2];
        }
    }
#pragma unroll
    for (int mi = 0; mi < MT; ++mi)
#pragma unroll
      for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int dd = mi * 16 + (lane >> 2) + (e >> 1) * 8, h = nt * 8 + (lane & 3) * 2 + (e & 1);
          sO[(warp * GMAX8 + h) * D + dd] = o[mi][nt][e];
        }
    __syncthreads();
    for (int e = tid; e < G * D; e += blockDim.x) {
      const int h = e / D, dd = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sWM[w * GMAX8 + h]);
      float L = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = fast_exp2(sWM[w * GMAX8 + h] - M);  // 0 for a warp that saw no rows
          L = fmaf(f, sWL[w * GMAX8 + h], L);
          acc = fmaf(f, sO[(w * GMAX8 + h) * D + dd], acc);
        }
      }
      const int64_t row = (int64_t)b * a.h_q + g * G + h;
      a.out[row * D + dd] = L > 0.f ? acc / L : 0.f;
      if (dd == 0 && a.lse) a.lse[row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
  }
};

// ---- Reading the row pack, bf16 ---------------------------------------------------------------
// The unit's packed chunks stream through kPackStages stages of (K tile, V tile), each tile one bulk
// copy of the chunk's rows, completed on an mbarrier; one block barrier per chunk (the stage's
// release).  Nothing leaves the block before the normalised output: no chunk partials, no merge pass.
constexpr int kPackStages = 2;

template <int D, int GMAX>
struct DraftPackCfg {
  static constexpr int ROWB = D * 2;
  static constexpr int CPR = ROWB / 16;
  static constexpr int TILE = kDraftChunk * ROWB;
  // [stages][K tile, V tile] (after the last chunk: the warps' outputs for the merge); the warps'
  // running max and sum [4][GMAX8] each; an mbarrier per stage.
  static constexpr int GMAX8 = DraftWarp<D, GMAX>::GMAX8;
  static constexpr int OFF_M = kPackStages * 2 * TILE;
  static constexpr int OFF_BAR = OFF_M + 2 * 4 * GMAX8 * 4;
  static constexpr int SMEM = OFF_BAR + kPackStages * 8;
  static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
  static_assert(4 * GMAX8 * D * 4 <= kPackStages * 2 * TILE, "merge area must fit in the stages");
};

template <int D, int GMAX>
__device__ __forceinline__ void draft_pack_unit(const DraftArgs &a, int unit, char *smem) {
  using C = DraftPackCfg<D, GMAX>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h_kv = a.kv.h_kv, b = unit / h_kv, g = unit % h_kv;
  const char *pu = a.pack + (int64_t)unit * a.C_max * (2 * C::TILE);
  // Before the wait for the previous kernel: the unit's first packed chunk (K and V tiles, whole)
  // into L2, so the first bulk copies after the wait find it there.  A prefetch only warms L2, which
  // every write also passes through, so it may overlap an earlier kernel still writing the pack.
  if (tid == 0) sm100::prefetch_l2(pu, 2 * C::TILE);
  pdl_wait();
  int n_all = a.cnt[unit];
  if (n_all < 0 || n_all > a.k_max) {
    if (tid == 0) atomicOr(a.status, (unsigned)SSD_FAULT_KMAX);
    n_all = n_all < 0 ? 0 : a.k_max;
  }
  const int nch = cdiv(n_all, kDraftChunk);  // 0 for an empty list
  float *sWM = reinterpret_cast<float *>(smem + C::OFF_M), *sWL = sWM + 4 * C::GMAX8;
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);

  // Chunk c's n rows of K and of V into stage c % kPackStages (thread 0).
  auto issue = [&](int c) {
    const int st = c % kPackStages;
    const uint32_t bytes = (uint32_t)(min(kDraftChunk, n_all - c * kDraftChunk) * C::ROWB);
    const uint32_t bar = bar0 + 8 * st;
    const char *src = pu + (int64_t)c * (2 * C::TILE);
    const uint32_t dst = smem_u32(smem + st * (2 * C::TILE));
    sm100::mbar_arrive_expect_tx(bar, 2 * bytes);
    sm100::bulk_load(dst, src, bytes, bar);
    sm100::bulk_load(dst + C::TILE, src + C::TILE, bytes, bar);
  };
  if (tid == 0) {
    for (int st = 0; st < kPackStages; ++st) sm100::mbar_init(bar0 + 8 * st, 1);
    sm100::mbar_init_fence();
    sm100::fence_proxy_async_smem();
    for (int c = 0; c < min(nch, kPackStages); ++c) issue(c);
  }
  DraftWarp<D, GMAX> W;
  W.init(a, b, g, lane);
  const int r0 = warp * 16;  // this warp's rows of every chunk
  int c_abort = -1;          // the chunk whose tiles did not land in time
  __syncthreads();           // barriers initialised

  for (int c = 0; c < nch; ++c) {
    const int st = c % kPackStages;
    const char *sKt = smem + st * (2 * C::TILE);
    char *sVt = smem + st * (2 * C::TILE) + C::TILE;
    const int n = min(kDraftChunk, n_all - c * kDraftChunk);
    // A thread whose wait expires still runs the chunk (on whatever the stage holds); the block
    // decides together at the stage barrier.
    const bool landed = draft_tile_wait(bar0 + 8 * st, (uint32_t)((c / kPackStages) & 1), a.status);
    // V rows past n (last chunk) of this warp's rows are zeroed: their P is 0, but 0 times a stale
    // non-finite value is not.  K rows past n need nothing: their logits are replaced by -inf.
    if (r0 + 16 > n)
      for (int e = lane; e < 16 * C::CPR; e += 32)
        if (r0 + e / C::CPR >= n)
          reinterpret_cast<uint4 *>(sVt + (r0 + e / C::CPR) * C::ROWB)[e % C::CPR] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    W.chunk(sKt, sVt, n, r0, a.scale_log2, lane);
    // Every warp is done with the stage (and the block learns whether a wait expired).
    if (__syncthreads_or(!landed)) {
      c_abort = c;
      break;
    }
    if (tid == 0 && c + kPackStages < nch) {
      sm100::fence_proxy_async_smem();  // the stage was read by every thread before the barrier
      issue(c + kPackStages);
    }
  }
  if (c_abort >= 0) {
    // A tile did not land in time (SSD_FAULT_TIMEOUT is set): no more copies are issued and the
    // unit's outputs are not written.  Thread 0 waits, bounded, for the copies still in flight into
    // this block's shared memory before the block exits; a copy that outlives that second wait too
    // means the device is unusable for this context.
    if (tid == 0)
      for (int cc = c_abort; cc < min(c_abort + kPackStages, nch); ++cc)
        draft_tile_wait(bar0 + 8 * (cc % kPackStages), (uint32_t)((cc / kPackStages) & 1), a.status);
    return;
  }
  pdl_trigger();
  if (a.pack_discard) {
    // The round's last read of the pack: its rows are in shared memory by now, so the unit's lines
    // (the stored rows of every chunk, K and V tiles) leave L2 without being written back.
    for (int c = 0; c < nch; ++c) {
      const int lines = min(kDraftChunk, n_all - c * kDraftChunk) * C::ROWB / 128;
      for (int e = tid; e < 2 * lines; e += blockDim.x)
        discard_l2_line(pu + (int64_t)c * (2 * C::TILE) + (e >= lines ? C::TILE : 0) + (int64_t)(e % lines) * 128);
    }
  }
  W.merge_store(a, b, g, reinterpret_cast<float *>(smem), sWM, sWL);
}

}  // namespace ssd
