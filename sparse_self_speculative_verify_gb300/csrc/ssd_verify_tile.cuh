// ssd_verify_tile.cuh -- one verify work item: a split of up to kSplitTokens tokens of one
// (request b, KV head g), all R = G * n_cand query rows of the group at once.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: verification computes full attention for the k+1 candidates and its
// kernel dumps the attention scores on the fly, caching logits and the log-sum-exp so that the
// scores can be rematerialised.  Here the "cached logits" are stored in a compact form: for every
// (row, token) the fp16 value e = 2^(s - m_ref) in (0, 1], where m_ref is the row's running maximum
// (log2 domain) when the token was processed, and m_ref itself once per (row, 16 tokens).  The
// finalize pass (ssd_verify.cu) turns them into probabilities with the row's global LSE:
// p = e * 2^(m_ref - LSE2).
//
// Tensor-core path (bf16, d = 64/128): 4 warps = NRT row tiles of 16 query rows x NTG token groups.
// The GQA group's R rows form the M side of the QK^T and PV tiles (m16n8k16 bf16 MMAs); K/V tiles of
// 64 tokens are staged into swizzled shared memory by 16-byte cp.async in a 3-deep ring; each warp
// keeps an online softmax for its rows over its tokens and the token groups are merged at the end
// of the item.  P enters PV as bf16 hi + bf16 residual (two MMAs), which keeps ~16 bits of the
// probability.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// Arguments of the finalize pass (LSE merge of a unit's splits, output combine, criticality).
struct FinalizeArgs {
  const int32_t *seq_lens;
  int max_seq_len, h_kv, h_q, n_c, G, R, D;
  int S_max, Lpad;
  const float *o_parts;
  const float *lse_parts;
  const __half *side_p;   // [units][R][Lpad]
  const float *side_m;    // [units][R][ref_stride(Lpad, ref_shift)]
  const int32_t *ucnt;    // block-sparse pass: splits per unit from the union size
  const int *split_len;   // split length the verify wrote (tensor-core, fp32 paths); nullptr = kSplitTokens;
                          // tensor-core path: [1] holds the first request of the half-length tail
  int balanced;           // splits cut by tc_split_count (the tensor-core verify), else cdiv(L, split length)
  int ref_shift = kRefShift;  // one reference per (1 << ref_shift) tokens: kTcRefShift from the tensor-core verify
  const uint8_t *phase;   // unified launch: units of draft-phase requests are skipped
  int umax;
  float *out;
  float *lse;
  float *scores;
  int64_t scores_stride;
  float *bscores;
  int64_t bstride;
  // Fused Top-K (nullptr ks: none): row u of the scores keeps K = min(ks[b], L_b) tokens, written
  // as the select pass writes them (sel_idx [units][sel_kmax], sel_cnt [units]).
  const int32_t *ks;
  int32_t *sel_idx;
  int32_t *sel_cnt;
  int sel_kmax;
  unsigned *sel_ctr;  // [units] arrivals of a unit's token blocks, in the counter area
  // Row pack (nullptr: none): the selected tokens' K and V rows, stored where the draft's pack reader
  // takes them ([unit][chunk of 64][K tile, V tile], rows in the draft's swizzled order).
  char *pack;
  int pack_cmax;  // chunks per unit
  int esize;      // bytes per cache element
  KVView kv;
  unsigned *status;
};
struct VerifyArgs {
  KVView kv;
  const void *q;  // [B][n_c][h_q][D]
  int h_q, n_c, G, R;
  float scale_log2;  // softmax scale * log2(e)
  int S_max;         // splits per unit in the partial arrays
  int Lpad;          // tokens per unit in the side buffers (multiple of kSideAlign)
  float *o_parts;    // [units][S_max][R][D], normalised by the split's own sum
  float *lse_parts;  // [units][S_max][R], natural log; -inf for an empty split
  __half *side_p;    // [units][R][Lpad], or nullptr (no criticality)
  float *side_m;     // [units][R][Lpad / kRefGroup] (the tensor-core verify: [units][R][ref_stride(Lpad, kTcRefShift)])
  // Block-sparse token source (union of candidate block sets); nullptr for contiguous splits.
  const int32_t *uidx;
  const uint32_t *umask;
  const int32_t *ucnt;
  int umax;
  unsigned *status;
  int *sched;  // [2] in the counter area: next-item counter and finished-block count (tensor-core
               // path); zero at launch, and the last block to finish returns both to zero
  int *split_out;  // tensor-core and fp32 paths: receives the split length used (read by the finalize);
                   // tensor-core path: [1] the first request cut into half-length splits
  const uint8_t *phase;  // tensor-core path: nullptr, or only requests with phase[b] == 1 get items
  int early_trigger;     // tensor-core path: let the next kernel launch at once (see ssd_unified.cu)
};

template <int D, int NRT>
struct VerifyMmaCfg {
  static constexpr int NTG = 4 / NRT;
  static constexpr int TW = kStageTokens / NTG;  // tokens per warp per stage
  static constexpr int CPR = D / 8;              // 16-byte chunks per bf16 row
  static constexpr int ROWS = 16 * NRT;
  static constexpr int NSTAGE = 3;
  static constexpr int TILE = kStageTokens * D * 2;  // bytes of one K or V stage tile
  static constexpr int RING = NSTAGE * 2 * TILE;
  static constexpr int QBYTES = ROWS * D * 2;
  static constexpr int MERGE = NTG * ROWS * (D + 2) * 4;  // O, m, l of every token group
  static_assert(MERGE <= RING, "merge area must fit in the stage ring");
  // The pool row of every token of the item, resolved once at the item's start (after Q): kept where
  // it leaves room for two blocks per SM (all shapes but d = 128 with four row tiles).
  static constexpr int ROWTAB_BYTES = kSplitTokens * 4 + 2 * kBlocksPerItem * 4;  // + stage bases, masks
  static constexpr bool ROWTAB = RING + QBYTES + ROWTAB_BYTES <= 113 * 1024;
  static constexpr int SMEM = RING + QBYTES + (ROWTAB ? ROWTAB_BYTES : 0);
};
static_assert(kSplitTokens == kBlocksPerItem * kStageTokens, "an item is at most kSplitTokens tokens either way");

// Number of work items (splits) of one unit.
__device__ __forceinline__ int verify_splits(int L, int split = kSplitTokens) { return cdiv(L, split); }

// Splits of the tensor-core verify.  A unit of L tokens is cut into whole 128-token tiles, then into
// ns = round(L / split_len) splits (at least one, at most kTcMaxSplitTiles tiles each) whose tile
// counts differ by at most one: no split is a short ragged tail.  A work item's pipeline latency
// (loads, logits, softmax, P V, epilogue) is hidden behind the tiles of a long item but not of a
// short one, so a split of one to three tiles costs about as much as one of ten.
constexpr int kTcTileTokens = 128;
constexpr int kTcMaxSplitTiles = 16;
// Split length of request b: the requests whose items are handed out last (b >= tail_from: the shortest
// suffix of the batch whose items fit in one wave of blocks) get splits of half the length (whole tiles,
// at least kSplitTokens), so the last items of a launch are short and the blocks run out of work
// closer together.
__device__ __forceinline__ int tc_tail_split(int split_len, int b, int tail_from) {
  return b < tail_from ? split_len : max(kSplitTokens, split_len / 2 / kTcTileTokens * kTcTileTokens);
}
__device__ __forceinline__ int tc_split_count(int L, int split_len) {
  const int T = cdiv(L, kTcTileTokens);
  if (T <= 0) return 0;
  int ns = (L + split_len / 2) / split_len;
  ns = max(ns, cdiv(T, kTcMaxSplitTiles));
  return min(max(ns, 1), T);
}
// Tokens [t0, t1) of split s of a unit of L tokens.
__device__ __forceinline__ void tc_split_range(int L, int split_len, int s, int &t0, int &t1) {
  const int T = cdiv(L, kTcTileTokens), ns = tc_split_count(L, split_len);
  const int base = T / ns, extra = T % ns;
  const int first = s * base + min(s, extra);
  t0 = first * kTcTileTokens;
  t1 = min((first + base + (s < extra ? 1 : 0)) * kTcTileTokens, L);
}
__device__ __forceinline__ int block_splits(int ucnt) { return cdiv(ucnt, kBlocksPerItem); }

template <int D, int NRT, bool BLOCKS>
__device__ __forceinline__ void verify_item_mma(const VerifyArgs &a, int unit, int split, char *smem) {
  using C = VerifyMmaCfg<D, NRT>;
  constexpr int NTG = C::NTG, TW = C::TW, CPR = C::CPR, ROWS = C::ROWS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rt = warp % NRT, tg = warp / NRT;
  const int gq = lane >> 2, tq = lane & 3;
  const int h_kv = a.kv.h_kv;
  const int b = unit / h_kv, g = unit % h_kv;
  const int G = a.G, R = a.R, n_c = a.n_c;
  const int L = effective_len(a.kv, b, n_c, a.status);

  // Stages of this item: contiguous tokens [t_begin, t_end) or the union blocks of the item.
  int t_begin = 0, t_end = L, n_stages, blk_first = 0;
  if (BLOCKS) {
    int nu = min(a.ucnt[unit], a.umax);
    blk_first = split * kBlocksPerItem;
    n_stages = min(kBlocksPerItem, nu - blk_first);
  } else {
    t_begin = split * kSplitTokens;
    t_end = min(t_begin + kSplitTokens, L);
    n_stages = cdiv(t_end - t_begin, kStageTokens);
  }
  if (n_stages <= 0) return;

  char *ring = smem;
  char *qs = smem + C::RING;
  const __nv_bfloat16 *pool = reinterpret_cast<const __nv_bfloat16 *>(a.kv.pool);
  const int64_t v_off = (int64_t)h_kv * a.kv.page_size * D;  // V row = K row + v_off elements

  auto stage_base = [&](int s) -> int {
    if (BLOCKS) {
      int blk = a.uidx[(int64_t)unit * a.umax + blk_first + s];
      return blk * kStageTokens;
    }
    return t_begin + s * kStageTokens;
  };
  auto stage_bits = [&](int s) -> uint32_t {
    return BLOCKS ? a.umask[(int64_t)unit * a.umax + blk_first + s] : 0xffffffffu;
  };

  const int lim = BLOCKS ? L : t_end;
  // Pool row of every token of the item (0xffffffff: zero-filled), resolved once before the first
  // copies: the union block ids (block-sparse items), then the page ids, two loads deep for the
  // whole item instead of per stage, where the threads that issue a stage's copies would otherwise
  // wait for them right before computing the stage before it.
  uint32_t *s_rows = reinterpret_cast<uint32_t *>(smem + C::RING + C::QBYTES);
  if constexpr (C::ROWTAB) {
    constexpr int PER = kSplitTokens / 128;
    int tk[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int j = tid + 128 * k;
      tk[k] = j < n_stages * kStageTokens ? stage_base(j / kStageTokens) + j % kStageTokens : -1;
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int j = tid + 128 * k, t = tk[k];
      uint32_t row = 0xffffffffu;
      if (j < n_stages * kStageTokens && t >= 0 && t < lim) {
        const int32_t p = __ldg(a.kv.page_table + (int64_t)b * a.kv.max_pages + (t >> a.kv.log2_ps));
        const int64_t r = (((int64_t)p * 2) * h_kv + g) * a.kv.page_size + (t & (a.kv.page_size - 1));
        if (p < 0 || (int64_t)p >= a.kv.num_pages || r >= 0xffffffffll)
          atomicOr(a.status, (unsigned)SSD_FAULT_PAGE);
        else
          row = (uint32_t)r;
      }
      if (j < kSplitTokens) s_rows[j] = row;
    }
    if (BLOCKS && tid < n_stages) {  // the stages' first tokens and candidate masks, for the compute
      s_rows[kSplitTokens + tid] = (uint32_t)stage_base(tid);
      s_rows[kSplitTokens + kBlocksPerItem + tid] = a.umask[(int64_t)unit * a.umax + blk_first + tid];
    }
    __syncthreads();
  }

  // Issue the cp.async copies of stage s into ring buffer `buf`.  Rows past L (and rows whose page
  // id is out of range) are zero-filled.
  auto load_stage = [&](int s, int buf) {
    const int base = C::ROWTAB ? 0 : stage_base(s);
    char *kt = ring + buf * 2 * C::TILE;
    char *vt = kt + C::TILE;
#pragma unroll
    for (int it = 0; it < kStageTokens * CPR / 128; ++it) {
      int c = it * 128 + tid;
      int row = c / CPR, ch = c % CPR;
      const __nv_bfloat16 *kr = nullptr;
      if constexpr (C::ROWTAB) {
        const uint32_t rw = s_rows[s * kStageTokens + row];
        if (rw != 0xffffffffu) kr = pool + (int64_t)rw * D;
      } else {
        const int t = base + row;
        if (t >= 0 && t < lim) kr = kv_row<D, __nv_bfloat16>(a.kv, b, 0, g, t, a.status);
      }
      uint32_t off = row * (D * 2) + swz_chunk(row, ch) * 16;
      cp_async16(smem_u32(kt + off), kr ? (const void *)(kr + ch * 8) : (const void *)pool, kr ? 16 : 0);
      cp_async16(smem_u32(vt + off), kr ? (const void *)(kr + v_off + ch * 8) : (const void *)pool, kr ? 16 : 0);
    }
  };

  // Prologue: start the first stages, then stage Q (rows >= R are zero).
#pragma unroll
  for (int s = 0; s < C::NSTAGE - 1; ++s) {
    if (s < n_stages) load_stage(s, s);
    cp_async_commit();
  }
  {
    const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    for (int c = tid; c < ROWS * CPR; c += 128) {
      int r = c / CPR, ch = c % CPR;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        int i = r / G, hl = r % G;
        const __nv_bfloat16 *src = q + (((int64_t)b * n_c + i) * a.h_q + g * G + hl) * D + ch * 8;
        v = __ldg(reinterpret_cast<const uint4 *>(src));
      }
      *reinterpret_cast<uint4 *>(qs + r * (D * 2) + swz_chunk(r, ch) * 16) = v;
    }
  }
  __syncthreads();
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    int mi = lane >> 3;
    int r = rt * 16 + (mi & 1) * 8 + (lane & 7);
    int ch = 2 * kk + (mi >> 1);
    ldsm_x4(smem_u32(qs + r * (D * 2) + swz_chunk(r, ch) * 16), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  // This thread's two rows and their visibility limits.
  const int r0 = rt * 16 + gq, r1 = r0 + 8;
  const int cand0 = r0 < R ? r0 / G : 0, cand1 = r1 < R ? r1 / G : 0;
  const int lim0 = r0 < R ? L - n_c + cand0 : L - 1;
  const int lim1 = r1 < R ? L - n_c + cand1 : L - 1;
  const bool st0 = r0 < R, st1 = r1 < R;

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  for (int s = 0; s < n_stages; ++s) {
    cp_async_wait<C::NSTAGE - 2>();
    __syncthreads();
    {
      int sn = s + C::NSTAGE - 1;
      if (sn < n_stages) load_stage(sn, sn % C::NSTAGE);
      cp_async_commit();
    }
    const char *kt = ring + (s % C::NSTAGE) * 2 * C::TILE;
    const char *vt = kt + C::TILE;
    const int base = BLOCKS && C::ROWTAB ? (int)s_rows[kSplitTokens + s] : stage_base(s);
    const uint32_t bits = BLOCKS && C::ROWTAB ? s_rows[kSplitTokens + kBlocksPerItem + s] : stage_bits(s);

    // S = Q K^T for this warp's 16 rows x TW tokens.
    float sacc[TW / 8][4];
#pragma unroll
    for (int n = 0; n < TW / 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < TW / 16; ++np) {
        int mi = lane >> 3;
        int r = tg * TW + np * 16 + (mi >> 1) * 8 + (lane & 7);
        int ch = 2 * kk + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(kt + r * (D * 2) + swz_chunk(r, ch) * 16), b0, b1, b2, b3);
        mma_bf16(sacc[2 * np], qa[kk], b0, b1);
        mma_bf16(sacc[2 * np + 1], qa[kk], b2, b3);
      }
    }

    // Scale into the log2 domain and mask tokens a row cannot see.
    const bool need_mask = BLOCKS || (base + kStageTokens - 1 > L - n_c);
    const bool vis0 = (bits >> cand0) & 1u, vis1 = (bits >> cand1) & 1u;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < TW / 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sacc[n][e] * a.scale_log2;
        if (need_mask) {
          int t = base + tg * TW + n * 8 + 2 * tq + (e & 1);
          bool ok = (e < 2) ? (t <= lim0 && (r0 >= R || vis0)) : (t <= lim1 && (r1 >= R || vis1));
          v = ok ? v : -INFINITY;
        }
        sacc[n][e] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(sacc[n][0], sacc[n][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[n][2], sacc[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = fast_exp2(m_run[0] - base0), al1 = fast_exp2(m_run[1] - base1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    l_run[0] *= al0;
    l_run[1] *= al1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }
#pragma unroll
    for (int n = 0; n < TW / 8; ++n) {
      sacc[n][0] = fast_exp2(sacc[n][0] - base0);
      sacc[n][1] = fast_exp2(sacc[n][1] - base0);
      sacc[n][2] = fast_exp2(sacc[n][2] - base1);
      sacc[n][3] = fast_exp2(sacc[n][3] - base1);
      l_run[0] += sacc[n][0] + sacc[n][1];
      l_run[1] += sacc[n][2] + sacc[n][3];
    }

    // Criticality side values: e = 2^(s - base) as fp16, and base once per 16 tokens.
    if (!BLOCKS && a.side_p != nullptr) {
      const int tw0 = base + tg * TW;
      __half *sp0 = a.side_p + ((int64_t)unit * R + r0) * a.Lpad + tw0 + 2 * tq;
      __half *sp1 = a.side_p + ((int64_t)unit * R + r1) * a.Lpad + tw0 + 2 * tq;
#pragma unroll
      for (int n = 0; n < TW / 8; ++n) {
        if (st0) *reinterpret_cast<uint32_t *>(sp0 + n * 8) = pack_half(sacc[n][0], sacc[n][1]);
        if (st1) *reinterpret_cast<uint32_t *>(sp1 + n * 8) = pack_half(sacc[n][2], sacc[n][3]);
      }
      if (tq == 0) {
        const int nref = a.Lpad / kRefGroup;
#pragma unroll
        for (int j = 0; j < TW / kRefGroup; ++j) {
          if (st0) a.side_m[((int64_t)unit * R + r0) * nref + tw0 / kRefGroup + j] = base0;
          if (st1) a.side_m[((int64_t)unit * R + r1) * nref + tw0 / kRefGroup + j] = base1;
        }
      }
    }

    // O += P V, with P = hi + lo (two bf16 MMAs).
#pragma unroll
    for (int kt2 = 0; kt2 < TW / 16; ++kt2) {
      uint32_t ah[4], alo[4];
      split_bf16(sacc[2 * kt2][0], sacc[2 * kt2][1], ah[0], alo[0]);
      split_bf16(sacc[2 * kt2][2], sacc[2 * kt2][3], ah[1], alo[1]);
      split_bf16(sacc[2 * kt2 + 1][0], sacc[2 * kt2 + 1][1], ah[2], alo[2]);
      split_bf16(sacc[2 * kt2 + 1][2], sacc[2 * kt2 + 1][3], ah[3], alo[3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        int mi = lane >> 3;
        int r = tg * TW + kt2 * 16 + (mi & 1) * 8 + (lane & 7);
        int ch = 2 * dp + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(vt + r * (D * 2) + swz_chunk(r, ch) * 16), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], ah, b0, b1);
        mma_bf16(o[2 * dp], alo, b0, b1);
        mma_bf16(o[2 * dp + 1], ah, b2, b3);
        mma_bf16(o[2 * dp + 1], alo, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // Merge the token groups of each row tile and write the split's normalised partial.
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
  l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
  l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
  __syncthreads();  // every warp is done with the ring
  float *mo = reinterpret_cast<float *>(ring);          // [NTG][ROWS][D]
  float *mm = mo + NTG * ROWS * D;                      // [NTG][ROWS]
  float *ml = mm + NTG * ROWS;                           // [NTG][ROWS]
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    int col = n * 8 + 2 * tq;
    *reinterpret_cast<float2 *>(mo + (tg * ROWS + r0) * D + col) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2 *>(mo + (tg * ROWS + r1) * D + col) = make_float2(o[n][2], o[n][3]);
  }
  if (tq == 0) {
    mm[tg * ROWS + r0] = m_run[0];
    mm[tg * ROWS + r1] = m_run[1];
    ml[tg * ROWS + r0] = l_run[0];
    ml[tg * ROWS + r1] = l_run[1];
  }
  __syncthreads();
  const int64_t prow = ((int64_t)unit * a.S_max + split) * R;
  for (int idx = tid; idx < R * D; idx += 128) {
    int r = idx / D, dd = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < NTG; ++t) M = fmaxf(M, mm[t * ROWS + r]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int t = 0; t < NTG; ++t) {
        float w = fast_exp2(mm[t * ROWS + r] - M);
        acc += w * mo[(t * ROWS + r) * D + dd];
        lsum += w * ml[t * ROWS + r];
      }
    }
    bool empty = !(lsum > 0.f);
    a.o_parts[(prow + r) * D + dd] = empty ? 0.f : acc / lsum;
    if (dd == 0) a.lse_parts[prow + r] = empty ? -INFINITY : (M + __log2f(lsum)) * kLn2;
  }
}

// ------------------------------------------------------------------------------------------------
// SIMT path for fp32 caches (any R <= 64, d = 64/128): exact fp32 dot products on CUDA cores.  The
// whole split's logits stay in shared memory, so the reference of the side values is the split's
// exact row maximum.
// ------------------------------------------------------------------------------------------------
template <int D>
struct VerifySimtCfg {
  static constexpr int CH = 64;  // tokens staged per step
  static constexpr int KSTR = D + 1;
  static constexpr int SMEM = (kMaxRows * D + kMaxRows * kSimtSplitTokens + CH * KSTR + 2 * kMaxRows) * 4;
};

template <int D>
__device__ __forceinline__ void verify_item_simt(const VerifyArgs &a, int unit, int split, char *smem) {
  using C = VerifySimtCfg<D>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h_kv = a.kv.h_kv;
  const int b = unit / h_kv, g = unit % h_kv;
  const int G = a.G, R = a.R, n_c = a.n_c;
  const int L = effective_len(a.kv, b, n_c, a.status);
  const int t0 = split * kSimtSplitTokens, t1 = min(t0 + kSimtSplitTokens, L);
  const int n = t1 - t0;
  if (n <= 0) return;
  float *sQ = reinterpret_cast<float *>(smem);  // [R][D]
  float *sS = sQ + kMaxRows * D;                 // [R][kSimtSplitTokens]
  float *sK = sS + kMaxRows * kSimtSplitTokens;  // [CH][D+1]
  float *sBase = sK + C::CH * C::KSTR;           // [R]
  float *sL = sBase + kMaxRows;                  // [R]
  const float *q = reinterpret_cast<const float *>(a.q);
  for (int e = tid; e < R * D; e += blockDim.x) {
    int r = e / D, dd = e % D, i = r / G, hl = r % G;
    sQ[e] = q[(((int64_t)b * n_c + i) * a.h_q + g * G + hl) * D + dd];
  }
  // Stages CH tokens of K (which = 0) or V (which = 1) into sK: every page lookup of the step is
  // issued before any row load, then every row load (16 bytes each) before any store, so a step
  // costs two memory latencies whatever the number of loads per thread.
  auto stage = [&](int c0, int which) {
    constexpr int V4 = D / 4, PER_T = C::CH * V4 / 128;
    static_assert(C::CH * V4 % 128 == 0, "whole 16-byte loads per thread");
    __syncthreads();
    const float *rows[PER_T];
#pragma unroll
    for (int k = 0; k < PER_T; ++k) {
      const int e = tid + k * 128, j = e / V4;
      rows[k] = (c0 + j < n) ? kv_row<D, float>(a.kv, b, which, g, t0 + c0 + j, a.status) : nullptr;
    }
    float4 v[PER_T];
#pragma unroll
    for (int k = 0; k < PER_T; ++k)
      v[k] = rows[k] ? __ldg(reinterpret_cast<const float4 *>(rows[k]) + (tid + k * 128) % V4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < PER_T; ++k) {
      const int e = tid + k * 128, j = e / V4, q4 = e % V4;
      float *dst = sK + j * C::KSTR + 4 * q4;
      dst[0] = v[k].x;
      dst[1] = v[k].y;
      dst[2] = v[k].z;
      dst[3] = v[k].w;
    }
    __syncthreads();
  };
  for (int c0 = 0; c0 < n; c0 += C::CH) {
    stage(c0, 0);
    for (int e = tid; e < R * C::CH; e += blockDim.x) {
      int r = e / C::CH, j = e % C::CH, t = t0 + c0 + j;
      float acc = 0.f;
      for (int dd = 0; dd < D; ++dd) acc = fmaf(sQ[r * D + dd], sK[j * C::KSTR + dd], acc);
      bool ok = (c0 + j < n) && (t <= L - n_c + r / G);
      if (c0 + j < kSimtSplitTokens) sS[r * kSimtSplitTokens + c0 + j] = ok ? acc * a.scale_log2 : -INFINITY;
    }
  }
  __syncthreads();
  // Row maxima and sums over the split.
  for (int r = warp; r < R; r += blockDim.x / 32) {
    float m = -INFINITY;
    for (int j = lane; j < n; j += 32) m = fmaxf(m, sS[r * kSimtSplitTokens + j]);
    m = warp_max(m);
    float base = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
    for (int j = lane; j < n; j += 32) {
      float p = fast_exp2(sS[r * kSimtSplitTokens + j] - base);
      sS[r * kSimtSplitTokens + j] = p;
      l += p;
    }
    l = warp_sum(l);
    if (lane == 0) {
      sBase[r] = m == -INFINITY ? -INFINITY : base;
      sL[r] = l;
    }
  }
  __syncthreads();
  if (a.side_p != nullptr) {
    const int nref = a.Lpad / kRefGroup;
    for (int e = tid; e < R * n; e += blockDim.x) {
      int r = e / n, j = e % n;
      a.side_p[((int64_t)unit * R + r) * a.Lpad + t0 + j] = __float2half_rn(sS[r * kSimtSplitTokens + j]);
    }
    for (int e = tid; e < R * cdiv(n, kRefGroup); e += blockDim.x) {
      int r = e / cdiv(n, kRefGroup), j = e % cdiv(n, kRefGroup);
      float bs = sBase[r];
      a.side_m[((int64_t)unit * R + r) * nref + t0 / kRefGroup + j] = bs == -INFINITY ? 0.f : bs;
    }
  }
  // O = P V, one output element per thread and pass.
  constexpr int PER = (kMaxRows * D + 127) / 128;
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  for (int c0 = 0; c0 < n; c0 += C::CH) {
    stage(c0, 1);
    const int jn = min(C::CH, n - c0);
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      int e = tid + k * 128;
      if (e < R * D) {
        int r = e / D, dd = e % D;
        float s = acc[k];
        for (int j = 0; j < jn; ++j) s = fmaf(sS[r * kSimtSplitTokens + c0 + j], sK[j * C::KSTR + dd], s);
        acc[k] = s;
      }
    }
  }
  const int64_t prow = ((int64_t)unit * a.S_max + split) * R;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    int e = tid + k * 128;
    if (e < R * D) {
      int r = e / D, dd = e % D;
      float l = sL[r];
      bool empty = !(l > 0.f);
      a.o_parts[(prow + r) * D + dd] = empty ? 0.f : acc[k] / l;
      if (dd == 0) a.lse_parts[prow + r] = empty ? -INFINITY : (sBase[r] + __log2f(l)) * kLn2;
    }
  }
}

constexpr int kFinThreads = 256;
constexpr int kFinTok = kFinThreads * 8;  // eight consecutive tokens per thread
constexpr int kFinGroups = kFinTok / kRefGroup;

// Launches the finalize pass: grid (n_tok + n_comb, units); implemented in ssd_verify.cu.
int launch_finalize(const FinalizeArgs &f, int n_tok, int units, cudaStream_t st);

}  // namespace ssd
