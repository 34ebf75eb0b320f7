// ssd_topk.cuh -- exact Top-K of one score row by one thread block (shared by the select kernels
// and the finalize's fused selection).
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: Top-K over the dumped, GQA-reduced verify scores gives the sparse pattern.
// An exact radix select on the order-preserving 32-bit key of each fp32 score (four 8-bit MSB-first
// histogram passes find the K-th largest key tau), then a stream compaction in index order that keeps
// every key > tau and the lowest-index keys == tau until K are kept: ties go to the lower index and
// the output comes out sorted.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

constexpr int kSelItems = 4;

// Order-preserving key: unsigned order of the keys = numeric order of the floats; -0.0 == +0.0.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one value per thread; *total receives the sum.
template <int NW>
__device__ __forceinline__ int block_excl_scan(int v, int *s_warp, int *s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < NW) s_warp[lane] = wi - w;
    if (lane == NW - 1) *s_total = wi;
  }
  __syncthreads();
  int res = s_warp[warp] + incl - v;
  __syncthreads();
  return res;
}

// Scratch of topk_row for an NT-thread block.
template <int NT>
struct TopkScratch {
  uint32_t hist[NT / 32][256];
  uint32_t tot[256];
  int wgt[NT / 32], weq[NT / 32];
  uint32_t digit;
  int rem;
};

// Writes the K (0 <= K <= n) largest of the n keys key(0..n-1) to out[0..K) in ascending index order
// (equal keys toward the lower index) and -1 to out[K..k_max).  Threads 0 .. NT-1 of the block call
// it; `key` must give every thread the same value for the same index; `sync` is a barrier over those
// NT threads (__syncthreads when they are the whole block).
//
// Warp w owns the keys [w seg, (w + 1) seg) (seg a multiple of 32); in each round its lanes read 32
// consecutive keys.  Four MSB-first 8-bit passes find the K-th largest key tau (per-warp shared
// histograms; the thread that sums a bin over the warps also clears it for the next pass; warp 0
// finds the digit), then each warp counts its keys > tau and == tau, every warp takes its prefix
// over the warps before it, and a second pass writes the kept indices in index order: every key
// > tau, and the keys == tau while fewer than the needed number of them lie before (ballots give
// the ranks within a round).  Fifteen block barriers per row.
template <int NT, typename KeyFn, typename SyncFn>
__device__ __forceinline__ void topk_row(KeyFn key, int n, int K, int32_t *out, int k_max, TopkScratch<NT> &sc,
                                         SyncFn sync) {
  static_assert(NT >= 256 && NT % 32 == 0, "one thread per histogram bin");
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  if (K == n) {
    for (int t = tid; t < n; t += NT) out[t] = t;
  } else if (K > 0) {
    const int seg = cdiv(cdiv(n, NW), 32) * 32;
    const int lo = min(warp * seg, n), hi = min(lo + seg, n);
    for (int e = tid; e < NW * 256; e += NT) (&sc.hist[0][0])[e] = 0u;
    sync();
    uint32_t prefix = 0, mask = 0;
    int rem = K;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      // Four keys per lane are loaded before their atomics, so the loads of a lane overlap (the
      // compiler cannot move them across the shared atomics itself).
      int t = lo + lane;
      for (; t + 96 < hi; t += 128) {
        uint32_t k[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) k[j] = key(t + 32 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((k[j] & mask) == prefix) atomicAdd(&sc.hist[warp][(k[j] >> shift) & 255u], 1u);
      }
      for (; t < hi; t += 32) {
        const uint32_t k = key(t);
        if ((k & mask) == prefix) atomicAdd(&sc.hist[warp][(k >> shift) & 255u], 1u);
      }
      sync();
      if (tid < 256) {
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          s += sc.hist[w][tid];
          sc.hist[w][tid] = 0u;
        }
        sc.tot[tid] = s;
      }
      sync();
      if (warp == 0) {
        // Lane l owns bins 255-8l .. 248-8l (descending).
        uint32_t c[8];
        uint32_t sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = sc.tot[255 - 8 * lane - j];
          sum += c[j];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const uint32_t excl = incl - sum;
        unsigned hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)rem);
        int f = __ffs(hit) - 1;
        if (lane == f) {
          uint32_t run = excl;
          for (int j = 0; j < 8; ++j) {
            if (run + c[j] >= (uint32_t)rem) {
              sc.digit = 255u - 8u * lane - j;
              sc.rem = rem - (int)run;
              break;
            }
            run += c[j];
          }
        }
      }
      sync();
      prefix |= sc.digit << shift;
      mask |= 0xffu << shift;
      rem = sc.rem;
    }
    const uint32_t tau = prefix;
    const int need_eq = rem;
    int cgt = 0, ceq = 0;
    for (int t0 = lo; t0 < hi; t0 += 32) {
      const int t = t0 + lane;
      const uint32_t k = t < hi ? key(t) : 0u;
      cgt += __popc(__ballot_sync(0xffffffffu, t < hi && k > tau));
      ceq += __popc(__ballot_sync(0xffffffffu, t < hi && k == tau));
    }
    if (lane == 0) {
      sc.wgt[warp] = cgt;
      sc.weq[warp] = ceq;
    }
    sync();
    int pgt = 0, peq = 0;
    for (int w = 0; w < warp; ++w) {
      pgt += sc.wgt[w];
      peq += sc.weq[w];
    }
    int run_eq = peq;                   // keys == tau before this round, whole row
    int pos = pgt + min(peq, need_eq);  // output slot of this warp's next kept key
    for (int t0 = lo; t0 < hi; t0 += 32) {
      const int t = t0 + lane;
      const uint32_t k = t < hi ? key(t) : 0u;
      const bool gt = t < hi && k > tau, eq = t < hi && k == tau;
      const unsigned meq = __ballot_sync(0xffffffffu, eq);
      const bool keep = gt || (eq && run_eq + __popc(meq & lt) < need_eq);
      const unsigned mk = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int p = pos + __popc(mk & lt);
        if (p < K) out[p] = t;
      }
      pos += __popc(mk);
      run_eq += __popc(meq);
    }
  }
  for (int j = K + tid; j < k_max; j += NT) out[j] = -1;
}

template <int NT, typename KeyFn>
__device__ __forceinline__ void topk_row(KeyFn key, int n, int K, int32_t *out, int k_max, TopkScratch<NT> &sc) {
  topk_row<NT>(key, n, K, out, k_max, sc, [] { __syncthreads(); });
}

}  // namespace ssd
