// ssd_verify.cu -- verify attention with fused criticality (the host entry points and the
// non-tcgen05 kernels; the tcgen05 kernel is in ssd_verify_tc.cu), the split-KV finalize (LSE
// combine + criticality rematerialisation + block max-pool, and optionally the fused Top-K), the
// block-sparse union pass and the public split combine.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1 PillarAttn: the verify kernel dumps the attention scores while it runs,
// caching logits and LSE to rematerialise them; scores are reduced over the GQA group's heads and
// the verify positions.  SpecSA post, "overlap-aware grouped query execution": candidates whose
// sparse layouts overlap run together so shared KV blocks are loaded once.  SparDA §2: fine scores
// are max-pooled onto the coarser selection grid.
#include "ssd_finalize.cuh"
#include "ssd_host.h"

namespace ssd {

// ------------------------------------------------------------------------------------------------
// Verify kernels: grid (split, unit); one work item per block.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ int clamp_len(const KVView &kv, int b) {
  int L = kv.seq_lens[b];
  return L < 0 ? 0 : (L > kv.max_seq_len ? kv.max_seq_len : L);
}

template <int D, int NRT, bool BLOCKS>
__global__ void __launch_bounds__(128, 2) verify_mma_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) char smem[];
  const int unit = blockIdx.y, split = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (BLOCKS) {
    int nu = min(max(a.ucnt[unit], 0), a.umax);
    if (split >= block_splits(nu)) return;
  } else {
    if (split >= verify_splits(clamp_len(a.kv, unit / a.kv.h_kv))) return;
  }
  verify_item_mma<D, NRT, BLOCKS>(a, unit, split, smem);
}

template <int D>
__global__ void __launch_bounds__(128) verify_simt_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) char smem[];
  const int unit = blockIdx.y, split = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.split_out = kSimtSplitTokens;  // for the finalize
  if (split >= verify_splits(clamp_len(a.kv, unit / a.kv.h_kv), kSimtSplitTokens)) return;
  verify_item_simt<D>(a, unit, split, smem);
}

// ------------------------------------------------------------------------------------------------
// Finalize: grid (n_tok + n_comb, unit).  Every block merges the unit's split LSEs per row (one warp
// per row, lanes over splits); blocks x >= n_tok combine the split outputs of kFinRows rows each
// (one float4 of d per thread, splits unrolled), blocks x < n_tok rematerialise the criticality of
// kFinTok tokens each: crit[t] = sum_r e[r][t] * 2^(m_ref[r][t/16] - LSE2_r).  A token block past
// the unit's length exits first; the others issue their first kFinAhead rows of side values and
// their reference values before the LSE merge (neither depends on it), so one memory latency
// covers the merge, the references and the first rows.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ int fin_rows_per_cta(int D) { return kFinThreads / (D / 4); }

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(FinalizeArgs f, int n_tok) {
  __shared__ float sLn[kMaxRows];
  __shared__ float sL2[kMaxRows];
  __shared__ __align__(16) float s_coef[kMaxRows * kFinGroups];
  const int tid = threadIdx.x, lane = tid & 31;
  const int u = blockIdx.y, b = u / f.h_kv, g = u % f.h_kv;
  pdl_wait();
  if (f.phase && f.phase[b] == 0) return;
  int L = f.seq_lens[b];
  L = L < 0 ? 0 : (L > f.max_seq_len ? f.max_seq_len : L);
  const bool tok = (int)blockIdx.x < n_tok;
  const int tb0 = blockIdx.x * kFinTok;
  if (tok && (!f.side_p || tb0 >= L)) return;
  if (f.ks && (int)blockIdx.x == n_tok && L == 0) {  // an empty row has no token block: select nothing
    for (int j = tid; j < f.sel_kmax; j += kFinThreads) f.sel_idx[(int64_t)u * f.sel_kmax + j] = -1;
    if (tid == 0) f.sel_cnt[u] = 0;
  }
  const int ns = fin_splits(f, u, L);
  const int64_t pbase = (int64_t)u * f.S_max * f.R;
  const int64_t rbase = (int64_t)u * f.R;
  const int nref = ref_stride(f.Lpad, f.ref_shift);
  const int ng = kFinTok >> f.ref_shift;  // reference groups per token block (128 or 16)

  // Early loads of a token block: its first rows of side values and its reference values.
  const int t0 = tb0 + tid * 8;
  const bool valid = tok && t0 < L;
  const bool fast = tok && f.bscores == nullptr;
  const __half *sp = tok ? f.side_p + rbase * f.Lpad + t0 : nullptr;
  uint4 raw[kFinAhead];
  if (fast) {
#pragma unroll
    for (int k = 0; k < kFinAhead; ++k)
      raw[k] = (valid && k < f.R) ? __ldg(reinterpret_cast<const uint4 *>(sp + (int64_t)k * f.Lpad)) : make_uint4(0, 0, 0, 0);
  }
  if (tok) {
    // References straight into the coefficient table (16 bytes = 4 groups per copy; a row's
    // references start 16-byte aligned since Lpad is a multiple of 128 tokens).  Groups at or past
    // L are not fetched: no stored score reads their coefficient.
    for (int e = tid; e < f.R * (ng / 4); e += kFinThreads) {
      const int r = e / (ng / 4), j4 = (e % (ng / 4)) * 4;
      if (tb0 + (j4 << f.ref_shift) < L)
        cp_async16(smem_u32(s_coef + r * ng + j4), f.side_m + (rbase + r) * nref + (tb0 >> f.ref_shift) + j4, 16);
    }
    cp_async_commit();
  }

  fin_lse_merge<kFinThreads / 32>(f, pbase, ns, sLn, sL2);
  __syncthreads();
  pdl_trigger();

  if (!tok) {
    const int tpr = f.D / 4, rpc = fin_rows_per_cta(f.D);
    const int n_comb = (int)gridDim.x - n_tok;
    fin_combine_rows(f, pbase, ns, sLn, b, g, ((int)blockIdx.x - n_tok) * rpc + tid / tpr, rpc * n_comb, tid % tpr);
    if (n_comb == 1) {  // this block read every partial of the unit
      __syncthreads();
      fin_discard_parts(f, pbase, ns, tid, kFinThreads);
    }
    return;
  }

  // Criticality: coef[r][j] = 2^(m_ref[r][group j] - LSE2_r) for the ng reference groups of this
  // block, then crit[t] = sum_r e[r][t] * coef[r][group of t], eight consecutive tokens per thread.
  cp_async_wait<0>();
  __syncthreads();
  for (int e = tid; e < f.R * ng; e += kFinThreads) {
    const float l2 = sL2[e / ng];
    s_coef[e] = (l2 == -INFINITY) ? 0.f : fast_exp2(s_coef[e] - l2);
  }
  __syncthreads();
  const int grp = (tid * 8) >> f.ref_shift;  // this thread's 8 tokens lie in one reference group
  float crit[8], cc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) crit[k] = cc[k] = 0.f;
  if (fast) {
#pragma unroll
    for (int k = 0; k < kFinAhead; ++k)
      if (k < f.R) fin_fma_row(raw[k], s_coef[k * ng + grp], crit);
    for (int r0 = kFinAhead; r0 < f.R; r0 += kFinAhead) {
#pragma unroll
      for (int k = 0; k < kFinAhead; ++k)
        raw[k] = (valid && r0 + k < f.R) ? __ldg(reinterpret_cast<const uint4 *>(sp + (int64_t)(r0 + k) * f.Lpad))
                                         : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < kFinAhead; ++k)
        if (r0 + k < f.R) fin_fma_row(raw[k], s_coef[(r0 + k) * ng + grp], crit);
    }
  } else {
    for (int i = 0; i < f.n_c; ++i) {
#pragma unroll 4
      for (int hl = 0; hl < f.G; ++hl) {
        const int r = i * f.G + hl;
        const uint4 rw = valid ? __ldg(reinterpret_cast<const uint4 *>(sp + (int64_t)r * f.Lpad)) : make_uint4(0, 0, 0, 0);
        fin_fma_row(rw, s_coef[r * ng + grp], cc);
      }
      // Candidate i's block maximum: 64 tokens = 8 lanes x 8 tokens.
      float m = cc[0];
#pragma unroll
      for (int k = 1; k < 8; ++k) m = fmaxf(m, cc[k]);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      if ((lane & 7) == 0 && valid) f.bscores[((int64_t)u * f.n_c + i) * f.bstride + t0 / kBlockTokens] = m;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        crit[k] += cc[k];
        cc[k] = 0.f;
      }
    }
  }
  if (f.scores && valid) {
    float *dst = f.scores + (int64_t)u * f.scores_stride + t0;
    if (t0 + 8 <= L && ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
      reinterpret_cast<float4 *>(dst)[0] = make_float4(crit[0], crit[1], crit[2], crit[3]);
      reinterpret_cast<float4 *>(dst)[1] = make_float4(crit[4], crit[5], crit[6], crit[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (t0 + k < L) dst[k] = crit[k];
    }
  }
  // This block's side values have been read for the last time: drop their L2 lines unwritten (rows
  // start 256-byte aligned; the verify wrote whole 128-token tiles, kFinTok is a multiple of them).
  __syncthreads();
  {
    const int lines = (min(tb0 + kFinTok, cdiv(L, kSideAlign) * kSideAlign) - tb0) / 64;
    for (int e = tid; e < f.R * lines; e += kFinThreads)
      discard_l2_line(f.side_p + (rbase + e / lines) * f.Lpad + tb0 + (e % lines) * 64);
  }
  if (!f.ks) return;

  // Fused selection: the last of the unit's token blocks to finish selects the unit's row (read
  // back through L2; the other blocks' scores are visible after their fence and the ticket).
  __threadfence();
  __syncthreads();  // also: s_coef is free for the selection scratch
  __shared__ unsigned s_sel_last;
  if (tid == 0) s_sel_last = atomicAdd(f.sel_ctr + u, 1u) == (unsigned)(cdiv(L, kFinTok) - 1);
  __syncthreads();
  if (!s_sel_last) return;
  __threadfence();
  int K = f.ks[b];
  K = K < 0 ? 0 : (K > L ? L : K);
  if (K > f.sel_kmax) {
    if (tid == 0) atomicOr(f.status, (unsigned)SSD_FAULT_KMAX);
    K = f.sel_kmax;
  }
  const float *row = f.scores + (int64_t)u * f.scores_stride;
  static_assert(sizeof(s_coef) >= sizeof(TopkScratch<kFinThreads>), "selection scratch");
  auto &sc = *reinterpret_cast<TopkScratch<kFinThreads> *>(s_coef);
  topk_row<kFinThreads>([&](int t) -> uint32_t { return score_key(__ldcg(row + t)); }, L, K,
                        f.sel_idx + (int64_t)u * f.sel_kmax, f.sel_kmax, sc);
  if (f.pack) {
    static_assert(sizeof(s_coef) >= kPackBatch * sizeof(int64_t), "row-offset scratch");
    __syncthreads();  // the selection is read back below; the selection scratch is reused
    pack_unit_rows<kFinThreads>(f, u, K, tid, reinterpret_cast<int64_t *>(s_coef));
  }
  if (tid == 0) {
    f.sel_cnt[u] = K;
    f.sel_ctr[u] = 0u;
  }
}

// ------------------------------------------------------------------------------------------------
// Criticality and Top-K of one unit per block, and the split combine: the pass after the verify in
// ssd_verify_select when a row of scores fits in shared memory.  Blocks [0, units): unit
// u = blockIdx.x merges its split LSEs, rematerialises its row of scores from the side values with
// exactly the finalize's arithmetic (same coefficients, rows summed in the same order, so the same
// bits), writes the row out and keeps its keys in shared memory, then selects its Top-K from there
// (topk_row_smem: ties to the lower index, ascending output).  Blocks [units, 2 units): the combine of
// unit blockIdx.x - units.  One pass over the side values replaces the finalize's token blocks,
// the separate select launch and its read of the scores.
// ------------------------------------------------------------------------------------------------
constexpr int kCsThreads = 512;
constexpr int kCsSmemRow = 40960;  // longest row kept in shared memory (160 KB of keys)

#ifdef SSD_VERIFY_TRACE
// Diagnostic build: per unit-block of the criticality pass, global-timer stamps [0] entry, [1] past the
// wait for the verify, [2] LSE merge done, [3] scores done, [4] Top-K done, [5] row pack done, [6] side
// values dropped from L2; and the Top-K's phases: [8] histogram of the keys' top 12 bits, [9] threshold
// bin found, [10] tau found, [11] indices written.
constexpr int kCsTraceUnits = 4096;
constexpr int kCsTraceSlots = 16;
__device__ unsigned long long g_cs_trace[kCsTraceUnits * kCsTraceSlots];
__device__ __forceinline__ unsigned long long cs_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define CS_STAMP(k) \
  do {              \
    if (tid == 0 && u < kCsTraceUnits) g_cs_trace[u * kCsTraceSlots + (k)] = cs_ns(); \
  } while (0)
#else
#define CS_STAMP(k) \
  do {              \
  } while (0)
#endif

__global__ void __launch_bounds__(kCsThreads, 2) crit_select_kernel(FinalizeArgs f, int units) {
  extern __shared__ __align__(16) uint32_t s_keys[];  // [max_seq_len] keys of the unit's scores
  __shared__ float sLn[kMaxRows], sL2[kMaxRows];
  __shared__ TopkScratch<kCsThreads> sc;
  __shared__ uint32_t s_cand[kTopkCand];
  const int tid = threadIdx.x;
  const bool comb = (int)blockIdx.x >= units;
  const int u = comb ? (int)blockIdx.x - units : (int)blockIdx.x;
  const int b = u / f.h_kv, g = u % f.h_kv;
  if (!comb) CS_STAMP(0);
  pdl_wait();
  if (!comb) CS_STAMP(1);
  int L = f.seq_lens[b];
  L = L < 0 ? 0 : (L > f.max_seq_len ? f.max_seq_len : L);
  const int ns = fin_splits(f, u, L);
  const int64_t pbase = (int64_t)u * f.S_max * f.R;
  fin_lse_merge<kCsThreads / 32>(f, pbase, ns, sLn, sL2);
  __syncthreads();
  if (!comb) CS_STAMP(2);
  if (comb) {
    pdl_trigger();
    const int tpr = f.D / 4;
    fin_combine_rows(f, pbase, ns, sLn, b, g, tid / tpr, kCsThreads / tpr, tid % tpr);
    __syncthreads();
    fin_discard_parts(f, pbase, ns, tid, kCsThreads);
    return;
  }
  fin_unit_scores<kCsThreads>(f, u, L, sL2, s_keys, tid);
  pdl_trigger();
  __syncthreads();
  CS_STAMP(3);
  int K = f.ks[b];
  K = K < 0 ? 0 : (K > L ? L : K);
  if (K > f.sel_kmax) {
    if (tid == 0) atomicOr(f.status, (unsigned)SSD_FAULT_KMAX);
    K = f.sel_kmax;
  }
  topk_row_smem<kCsThreads>(s_keys, L, K, f.sel_idx + (int64_t)u * f.sel_kmax, f.sel_kmax, sc, s_cand, false,
                            [&](int k) { CS_STAMP(8 + k); });
  if (tid == 0) f.sel_cnt[u] = K;
  CS_STAMP(4);
  if (f.pack) {
    static_assert(sizeof(sc) >= kPackBatch * sizeof(int64_t), "row-offset scratch");
    __syncthreads();  // the selection, written by the whole block, is read back below
    pack_unit_rows<kCsThreads>(f, u, K, tid, reinterpret_cast<int64_t *>(&sc));
  }
  CS_STAMP(5);
  // The unit's side values were read for the last time before the Top-K: drop their L2 lines unwritten
  // (each row of the unit starts 256-byte aligned; the verify wrote whole 128-token tiles).  Issued
  // last, so that no barrier of the block waits for them.
  if (f.side_p) {
    const int lines = cdiv(L, kSideAlign) * kSideAlign / 64;  // 64 fp16 per 128-byte line
    for (int e = tid; e < f.R * lines; e += kCsThreads)
      discard_l2_line(f.side_p + ((int64_t)u * f.R + e / lines) * f.Lpad + (e % lines) * 64);
  }
  CS_STAMP(6);
}

#ifdef SSD_VERIFY_TRACE
// Diagnostic build only: the criticality-pass record (kCsTraceUnits x 8 64-bit words).
extern "C" int ssd_crit_select_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(g_cs_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, g_cs_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
#endif

int launch_finalize(const FinalizeArgs &f, int n_tok, int units, cudaStream_t st) {
  // With token blocks in the grid, one combine block per unit loops over the rows (fewer blocks to
  // schedule behind the token work); without them, a block per group of rows.
  const int n_comb = n_tok > 0 ? 1 : cdiv(f.R, kFinThreads / (f.D / 4));
  return launch(finalize_kernel, dim3(n_tok + n_comb, units), dim3(kFinThreads), 0, st, "finalize_kernel", f, n_tok);
}

// Public split combine: one block per row.
__global__ void __launch_bounds__(128) combine_kernel(const float *o_parts, const float *lse_parts, int n_splits,
                                                     int d, float *out, float *lse) {
  const int row = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  const float *lp = lse_parts + (int64_t)row * n_splits;
  float M = -INFINITY;
  for (int j = 0; j < n_splits; ++j) M = fmaxf(M, lp[j]);
  float s = 0.f;
  if (M != -INFINITY)
    for (int j = 0; j < n_splits; ++j) s += fast_exp2((lp[j] - M) * kLog2e);
  const float ln = (M == -INFINITY) ? -INFINITY : M + __logf(s);
  for (int dd = threadIdx.x; dd < d; dd += blockDim.x) {
    float acc = 0.f;
    if (ln != -INFINITY)
      for (int j = 0; j < n_splits; ++j)
        acc = fmaf(fast_exp2((lp[j] - ln) * kLog2e), o_parts[((int64_t)row * n_splits + j) * d + dd], acc);
    out[(int64_t)row * d + dd] = acc;
  }
  if (threadIdx.x == 0 && lse) lse[row] = ln;
}

// ------------------------------------------------------------------------------------------------
// Host side.
// ------------------------------------------------------------------------------------------------
bool verify_tc_supported(const ssd_paged_kv *kv, int R);
int launch_verify_tc(const ssd_paged_kv *kv, const VerifyArgs &a, cudaStream_t st, int max_blocks = 0);

static int rows_per_tile(int R) { return R <= 16 ? 1 : (R <= 32 ? 2 : 4); }

template <int D, int NRT, bool BLOCKS>
static int launch_mma(const VerifyArgs &a, dim3 grid, cudaStream_t st) {
  constexpr int smem = VerifyMmaCfg<D, NRT>::SMEM;
  int rc = ensure_smem<verify_mma_kernel<D, NRT, BLOCKS>>(smem);
  if (rc) return rc;
  return launch(verify_mma_kernel<D, NRT, BLOCKS>, grid, dim3(128), smem, st, "verify_mma_kernel", a);
}

template <bool BLOCKS>
static int dispatch_mma(int D, int NRT, const VerifyArgs &a, dim3 grid, cudaStream_t st) {
  if (D == 128) {
    if (NRT == 1) return launch_mma<128, 1, BLOCKS>(a, grid, st);
    if (NRT == 2) return launch_mma<128, 2, BLOCKS>(a, grid, st);
    return launch_mma<128, 4, BLOCKS>(a, grid, st);
  }
  if (NRT == 1) return launch_mma<64, 1, BLOCKS>(a, grid, st);
  if (NRT == 2) return launch_mma<64, 2, BLOCKS>(a, grid, st);
  return launch_mma<64, 4, BLOCKS>(a, grid, st);
}

template <int D>
static int launch_simt(const VerifyArgs &a, dim3 grid, cudaStream_t st) {
  constexpr int smem = VerifySimtCfg<D>::SMEM;
  int rc = ensure_smem<verify_simt_kernel<D>>(smem);
  if (rc) return rc;
  return launch(verify_simt_kernel<D>, grid, dim3(128), smem, st, "verify_simt_kernel", a);
}

struct VerifyLayout {
  int G, R, units, S_max, Lpad;
  size_t o_off, lse_off, sp_off, sm_off, split_off, ctr_off, total;
};

static VerifyLayout verify_layout(const ssd_paged_kv *kv, int h_q, int n_cand, int S_max) {
  VerifyLayout l{};
  l.G = h_q / kv->h_kv;
  l.R = l.G * n_cand;
  l.units = kv->batch * kv->h_kv;
  l.S_max = S_max;
  l.Lpad = cdiv(kv->max_seq_len > 0 ? kv->max_seq_len : 1, kSideAlign) * kSideAlign;
  Carver c(nullptr);
  l.ctr_off = c.off;  // counter area (item counter of the tensor-core kernel)
  c.take<unsigned>(kCounterSlots);
  size_t rows = (size_t)l.units * l.S_max * l.R;
  l.o_off = c.off;
  c.take<float>(rows * kv->d);
  l.lse_off = c.off;
  c.take<float>(rows);
  l.sp_off = c.off;
  c.take<__half>((size_t)l.units * l.R * l.Lpad);
  l.sm_off = c.off;
  c.take<float>((size_t)l.units * l.R * (l.Lpad / kRefGroup));
  l.split_off = c.off;
  c.take<int>(2);  // split length, first request of the half-length tail
  l.total = c.off;
  return l;
}

// Splits per unit the workspace holds: 512-token splits (the tensor-core verify picks longer ones),
// 128-token splits on the fp32 path.
static int verify_smax(const ssd_paged_kv *kv) {
  return cdiv(kv->max_seq_len, kv->dtype == SSD_DTYPE_F32 ? kSimtSplitTokens : kSplitTokens);
}

static int verify_common_checks(const ssd_paged_kv *kv, int h_q, int n_cand, const void *q, const float *out,
                                const char *who) {
  if (!q || !out) return fail(SSD_ERR_INVALID_ARG, "%s: q and out must be non-NULL", who);
  if (h_q <= 0 || h_q % kv->h_kv) return fail(SSD_ERR_INVALID_ARG, "%s: h_q %d not a multiple of h_kv %d", who, h_q, kv->h_kv);
  if (n_cand < 1) return fail(SSD_ERR_INVALID_ARG, "%s: n_cand %d < 1", who, n_cand);
  if ((h_q / kv->h_kv) * n_cand > kMaxRows)
    return fail(SSD_ERR_UNSUPPORTED, "%s: G*n_cand = %d exceeds %d", who, (h_q / kv->h_kv) * n_cand, kMaxRows);
  if (!aligned16(q) || !aligned16(out)) return fail(SSD_ERR_INVALID_ARG, "%s: q and out must be 16-byte aligned", who);
  if ((int64_t)kv->batch * kv->h_kv > 65535) return fail(SSD_ERR_UNSUPPORTED, "%s: batch*h_kv above 65535", who);
  return SSD_OK;
}

}  // namespace ssd

using namespace ssd;

extern "C" size_t ssd_verify_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand) {
  if (!kv || kv->h_kv <= 0 || h_q <= 0 || n_cand <= 0 || kv->batch < 0 || kv->max_seq_len < 0) return 0;
  return verify_layout(kv, h_q, n_cand, verify_smax(kv)).total;
}

static int verify_call(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                       float *lse, float *scores, int64_t scores_stride, float *bscores, int64_t bscores_stride,
                       int block_size, const int32_t *ks, int32_t *idx, int k_max, int32_t *cnt, void *pack,
                       size_t pack_bytes, void *workspace, size_t workspace_bytes, ssd_stream_t stream,
                       const char *who) {
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if ((rc = verify_common_checks(kv, h_q, n_cand, q, out, who))) return rc;
  if (scores && scores_stride < kv->max_seq_len)
    return fail(SSD_ERR_INVALID_ARG, "%s: scores_stride %lld < max_seq_len %d", who, (long long)scores_stride, kv->max_seq_len);
  if (bscores) {
    if (block_size != kBlockTokens) return fail(SSD_ERR_UNSUPPORTED, "%s: block_size %d (only 64)", who, block_size);
    if (bscores_stride < cdiv(kv->max_seq_len, kBlockTokens))
      return fail(SSD_ERR_INVALID_ARG, "%s: bscores_stride too small", who);
  }
  const VerifyLayout lay = verify_layout(kv, h_q, n_cand, verify_smax(kv));
  if (!workspace || workspace_bytes < lay.total)
    return fail(SSD_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", who, workspace_bytes, lay.total);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (ks) {
    if (!scores || bscores) return fail(SSD_ERR_INVALID_ARG, "%s: needs scores and no block scores", who);
    if (!cnt || (!idx && k_max > 0) || k_max < 0) return fail(SSD_ERR_INVALID_ARG, "%s: idx / cnt / k_max", who);
    if ((int64_t)kv->batch * kv->h_kv > kCounterSlots - 2)
      return fail(SSD_ERR_UNSUPPORTED, "%s: batch*h_kv above %d", who, kCounterSlots - 2);
  }
  if (pack) {
    const size_t pneed = ssd_draft_pack_bytes(kv, k_max);
    if (!ks || pneed == 0 || pack_bytes < pneed)
      return fail(SSD_ERR_WORKSPACE, "%s: row pack %zu bytes, need %zu", who, pack_bytes, pneed);
    if (reinterpret_cast<uintptr_t>(pack) & 255u)
      return fail(SSD_ERR_INVALID_ARG, "%s: row pack must be 256-byte aligned", who);
  }
  if (kv->batch == 0 || kv->max_seq_len == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  const bool crit = scores || bscores;

  VerifyArgs a{};
  a.kv = v;
  a.q = q;
  a.h_q = h_q;
  a.n_c = n_cand;
  a.G = lay.G;
  a.R = lay.R;
  a.scale_log2 = scale * kLog2e;
  a.S_max = lay.S_max;
  a.Lpad = lay.Lpad;
  a.o_parts = reinterpret_cast<float *>(ws + lay.o_off);
  a.lse_parts = reinterpret_cast<float *>(ws + lay.lse_off);
  a.side_p = crit ? reinterpret_cast<__half *>(ws + lay.sp_off) : nullptr;
  a.side_m = crit ? reinterpret_cast<float *>(ws + lay.sm_off) : nullptr;
  a.status = status;
  a.sched = reinterpret_cast<int *>(ws + lay.ctr_off);
  dim3 grid(lay.S_max, lay.units);
  const bool tc = verify_tc_supported(kv, lay.R);
  const bool simt = !tc && kv->dtype != SSD_DTYPE_BF16;
  a.split_out = reinterpret_cast<int *>(ws + lay.split_off);

  FinalizeArgs f{};
  f.seq_lens = kv->seq_lens;
  f.max_seq_len = kv->max_seq_len;
  f.h_kv = kv->h_kv;
  f.h_q = h_q;
  f.n_c = n_cand;
  f.G = lay.G;
  f.R = lay.R;
  f.D = kv->d;
  f.S_max = lay.S_max;
  f.Lpad = lay.Lpad;
  f.o_parts = a.o_parts;
  f.lse_parts = a.lse_parts;
  f.side_p = a.side_p;
  f.side_m = a.side_m;
  f.out = out;
  f.lse = lse;
  f.scores = scores;
  f.scores_stride = scores_stride;
  f.bscores = bscores;
  f.bstride = bscores_stride;
  f.split_len = (tc || simt) ? a.split_out : nullptr;
  f.balanced = tc ? 1 : 0;
  f.ref_shift = tc ? kTcRefShift : kRefShift;
  f.ks = ks;
  f.sel_idx = idx;
  f.sel_cnt = cnt;
  f.sel_kmax = k_max;
  f.sel_ctr = reinterpret_cast<unsigned *>(ws + lay.ctr_off) + 2;  // slots 0-1: the tensor-core kernel
  f.pack = static_cast<char *>(pack);
  f.pack_cmax = cdiv(k_max > 0 ? k_max : 1, kDraftChunk);
  f.esize = kv->dtype == SSD_DTYPE_BF16 ? 2 : 4;
  f.kv = v;
  f.status = status;

  if (tc) {
    rc = launch_verify_tc(kv, a, st);
  }
  else if (kv->dtype == SSD_DTYPE_BF16)
    rc = dispatch_mma<false>(kv->d, rows_per_tile(lay.R), a, grid, st);
  else
    rc = kv->d == 128 ? launch_simt<128>(a, grid, st) : launch_simt<64>(a, grid, st);
  if (rc) return rc;
  if (ks && kv->max_seq_len <= kCsSmemRow) {
    const int smem = kv->max_seq_len * 4;
    if ((rc = ensure_smem<crit_select_kernel>(smem))) return rc;
    return launch(crit_select_kernel, dim3(2 * lay.units), dim3(kCsThreads), smem, st, "crit_select_kernel", f,
                  lay.units);
  }
  const int n_tok = crit ? cdiv(kv->max_seq_len, kFinTok) : 0;
  return launch_finalize(f, n_tok, lay.units, st);
}

extern "C" int ssd_verify_attn(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                               float *lse, float *scores, int64_t scores_stride, float *bscores,
                               int64_t bscores_stride, int block_size, void *workspace, size_t workspace_bytes,
                               ssd_stream_t stream) {
  return verify_call(kv, q, h_q, n_cand, scale, out, lse, scores, scores_stride, bscores, bscores_stride, block_size,
                     nullptr, nullptr, 0, nullptr, nullptr, 0, workspace, workspace_bytes, stream, "ssd_verify_attn");
}

extern "C" int ssd_verify_select(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                                 float *lse, float *scores, int64_t scores_stride, const int32_t *ks, int32_t *idx,
                                 int k_max, int32_t *cnt, void *workspace, size_t workspace_bytes,
                                 ssd_stream_t stream) {
  const char *who = "ssd_verify_select";
  if (!ks) return fail(SSD_ERR_INVALID_ARG, "%s: ks must be non-NULL", who);
  return verify_call(kv, q, h_q, n_cand, scale, out, lse, scores, scores_stride, nullptr, 0, kBlockTokens, ks, idx,
                     k_max, cnt, nullptr, 0, workspace, workspace_bytes, stream, who);
}

extern "C" int ssd_verify_select_packed(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale,
                                        float *out, float *lse, float *scores, int64_t scores_stride,
                                        const int32_t *ks, int32_t *idx, int k_max, int32_t *cnt, void *pack,
                                        size_t pack_bytes, void *workspace, size_t workspace_bytes,
                                        ssd_stream_t stream) {
  const char *who = "ssd_verify_select_packed";
  if (!ks) return fail(SSD_ERR_INVALID_ARG, "%s: ks must be non-NULL", who);
  if (!pack) return fail(SSD_ERR_INVALID_ARG, "%s: pack must be non-NULL", who);
  return verify_call(kv, q, h_q, n_cand, scale, out, lse, scores, scores_stride, nullptr, 0, kBlockTokens, ks, idx,
                     k_max, cnt, pack, pack_bytes, workspace, workspace_bytes, stream, who);
}

extern "C" size_t ssd_block_sparse_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand, int umax) {
  if (!kv || kv->h_kv <= 0 || h_q <= 0 || n_cand <= 0 || umax <= 0 || kv->batch < 0) return 0;
  const int G = h_q / kv->h_kv, R = G * n_cand;
  const size_t rows = (size_t)kv->batch * kv->h_kv * cdiv(umax, kBlocksPerItem) * R;
  Carver c(nullptr);
  c.take<float>(rows * kv->d);
  c.take<float>(rows);
  return c.off;
}

extern "C" int ssd_block_sparse_attn(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, const int32_t *uidx,
                                     const uint32_t *umask, const int32_t *ucnt, int umax, int block_size, float scale,
                                     float *out, float *lse, void *workspace, size_t workspace_bytes,
                                     ssd_stream_t stream) {
  const char *who = "ssd_block_sparse_attn";
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if ((rc = verify_common_checks(kv, h_q, n_cand, q, out, who))) return rc;
  if (kv->dtype != SSD_DTYPE_BF16) return fail(SSD_ERR_UNSUPPORTED, "%s: bf16 caches only", who);
  if (block_size != kBlockTokens) return fail(SSD_ERR_UNSUPPORTED, "%s: block_size %d (only 64)", who, block_size);
  if (n_cand > 32) return fail(SSD_ERR_UNSUPPORTED, "%s: n_cand %d > 32", who, n_cand);
  if (!uidx || !umask || !ucnt || umax <= 0) return fail(SSD_ERR_INVALID_ARG, "%s: union arrays / umax", who);
  const size_t need = ssd_block_sparse_workspace_bytes(kv, h_q, n_cand, umax);
  if (!workspace || workspace_bytes < need)
    return fail(SSD_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", who, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (kv->batch == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int G = h_q / kv->h_kv, R = G * n_cand, units = kv->batch * kv->h_kv;
  const int S_max = cdiv(umax, kBlocksPerItem);
  Carver c(workspace);
  VerifyArgs a{};
  a.kv = v;
  a.q = q;
  a.h_q = h_q;
  a.n_c = n_cand;
  a.G = G;
  a.R = R;
  a.scale_log2 = scale * kLog2e;
  a.S_max = S_max;
  a.Lpad = 0;
  a.o_parts = c.take<float>((size_t)units * S_max * R * kv->d);
  a.lse_parts = c.take<float>((size_t)units * S_max * R);
  a.uidx = uidx;
  a.umask = umask;
  a.ucnt = ucnt;
  a.umax = umax;
  a.status = status;
  rc = dispatch_mma<true>(kv->d, rows_per_tile(R), a, dim3(S_max, units), st);
  if (rc) return rc;
  FinalizeArgs f{};
  f.seq_lens = kv->seq_lens;
  f.max_seq_len = kv->max_seq_len;
  f.h_kv = kv->h_kv;
  f.h_q = h_q;
  f.n_c = n_cand;
  f.G = G;
  f.R = R;
  f.D = kv->d;
  f.S_max = S_max;
  f.o_parts = a.o_parts;
  f.lse_parts = a.lse_parts;
  f.ucnt = ucnt;
  f.umax = umax;
  f.out = out;
  f.lse = lse;
  return launch_finalize(f, 0, units, st);
}

extern "C" int ssd_combine(const float *o_parts, const float *lse_parts, int n_rows, int n_splits, int d, float *out,
                           float *lse, ssd_stream_t stream) {
  if (n_rows < 0 || n_splits < 0 || d <= 0) return fail(SSD_ERR_INVALID_ARG, "ssd_combine: bad sizes");
  if (!out || (n_splits > 0 && (!o_parts || !lse_parts)))
    return fail(SSD_ERR_INVALID_ARG, "ssd_combine: NULL pointer");
  if (n_rows == 0) return SSD_OK;
  if (n_rows > (1 << 30)) return fail(SSD_ERR_UNSUPPORTED, "ssd_combine: too many rows");
  return launch(combine_kernel, dim3(n_rows), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream), "combine_kernel",
                o_parts, lse_parts, n_splits, d, out, lse);
}
