// ssd_topk.cuh -- exact Top-K of one score row by one thread block (shared by the select kernels
// and the finalize's fused selection).
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: Top-K over the dumped, GQA-reduced verify scores gives the sparse pattern.
// An exact radix select on the order-preserving 32-bit key of each fp32 score (MSB-first histogram
// passes find the K-th largest key tau), then a stream compaction in index order that keeps
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
  alignas(16) uint32_t hist[NT / 32][256];
  uint32_t tot[256];
  int wgt[NT / 32], weq[NT / 32];
  uint32_t digit;
  int rem;
  int cbin, ncand;
};

// Warp-wide: the bin of a 256-bin histogram (scanned from the top bin down) that holds the rem-th
// largest counted key, and that key's rank within its bin; every lane receives both.  Lane l owns
// bins 255 - 8l .. 248 - 8l.  The histogram counts at least rem keys.
__device__ __forceinline__ void warp_find_digit(const uint32_t *hist, int rem, uint32_t &digit, int &rem_in_bin) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[255 - 8 * lane - j];
    sum += c[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const int f = __ffs(__ballot_sync(0xffffffffu, incl >= (uint32_t)rem)) - 1;
  uint32_t d = 0;
  int r = 0;
  if (lane == f) {
    uint32_t run = incl - sum;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (run + c[j] >= (uint32_t)rem) {
        d = 255u - 8u * lane - j;
        r = rem - (int)run;
        break;
      }
      run += c[j];
    }
  }
  digit = __shfl_sync(0xffffffffu, d, f);
  rem_in_bin = __shfl_sync(0xffffffffu, r, f);
}

// One MSB-first 8-bit radix pass over warp w's keys [lo, hi) that match `prefix` on `mask`: per-warp
// histograms of bits [shift, shift + 8), summed per bin (the summing thread clears the bin for the
// next pass), then warp 0 finds the digit.  Narrows (prefix, mask, rem) to the digit's bin.  The
// per-warp histograms start zeroed.
template <int NT, typename KeyFn, typename SyncFn>
__device__ __forceinline__ void topk_block_pass(KeyFn key, int lo, int hi, int shift, uint32_t &prefix, uint32_t &mask,
                                                int &rem, TopkScratch<NT> &sc, SyncFn sync) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Four keys per lane are loaded before their atomics, so the loads of a lane overlap (the compiler
  // cannot move them across the shared atomics itself).
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
    uint32_t d;
    int r;
    warp_find_digit(sc.tot, rem, d, r);
    if (lane == 0) {
      sc.digit = d;
      sc.rem = r;
    }
  }
  sync();
  prefix |= sc.digit << shift;
  mask |= 0xffu << shift;
  rem = sc.rem;
}

// Given the K-th largest key tau, the number need_eq of keys == tau that are kept, and warp w's counts of
// its keys > tau (cgt) and == tau (ceq), each warp takes its prefix over the warps before it and writes
// its kept indices in index order: every key > tau, and the keys == tau while fewer than need_eq of
// them lie before (ballots give the ranks within a round of 32 keys).
template <int NT, typename KeyFn, typename SyncFn>
__device__ __forceinline__ void topk_emit_counted(KeyFn key, int lo, int hi, int K, uint32_t tau, int need_eq,
                                                  int cgt, int ceq, int32_t *out, TopkScratch<NT> &sc, SyncFn sync) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
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
#pragma unroll 4
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

// topk_emit_counted after a pass in which each warp counts its keys > tau and == tau.
template <int NT, typename KeyFn, typename SyncFn>
__device__ __forceinline__ void topk_emit(KeyFn key, int lo, int hi, int K, uint32_t tau, int need_eq, int32_t *out,
                                          TopkScratch<NT> &sc, SyncFn sync) {
  const int lane = threadIdx.x & 31;
  int cgt = 0, ceq = 0;
#pragma unroll 4
  for (int t0 = lo; t0 < hi; t0 += 32) {
    const int t = t0 + lane;
    const uint32_t k = t < hi ? key(t) : 0u;
    cgt += __popc(__ballot_sync(0xffffffffu, t < hi && k > tau));
    ceq += __popc(__ballot_sync(0xffffffffu, t < hi && k == tau));
  }
  topk_emit_counted<NT>(key, lo, hi, K, tau, need_eq, cgt, ceq, out, sc, sync);
}

// Writes the K (0 <= K <= n) largest of the n keys key(0..n-1) to out[0..K) in ascending index order
// (equal keys toward the lower index) and -1 to out[K..k_max).  Threads 0 .. NT-1 of the block call
// it; `key` must give every thread the same value for the same index; `sync` is a barrier over those
// NT threads (__syncthreads when they are the whole block).
//
// Warp w owns the keys [w seg, (w + 1) seg) (seg a multiple of 32); in each round its lanes read 32
// consecutive keys.  Four MSB-first 8-bit passes (topk_block_pass) find the K-th largest key tau,
// then topk_emit writes the kept indices.  Fifteen block barriers per row.
template <int NT, typename KeyFn, typename SyncFn>
__device__ __forceinline__ void topk_row(KeyFn key, int n, int K, int32_t *out, int k_max, TopkScratch<NT> &sc,
                                         SyncFn sync) {
  static_assert(NT >= 256 && NT % 32 == 0, "one thread per histogram bin");
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (K == n) {
    for (int t = tid; t < n; t += NT) out[t] = t;
  } else if (K > 0) {
    const int seg = cdiv(cdiv(n, NW), 32) * 32;
    const int lo = min(warp * seg, n), hi = min(lo + seg, n);
    for (int e = tid; e < NW * 256; e += NT) (&sc.hist[0][0])[e] = 0u;
    sync();
    uint32_t prefix = 0, mask = 0;
    int rem = K;
    for (int pass = 0; pass < 4; ++pass) topk_block_pass<NT>(key, lo, hi, 24 - 8 * pass, prefix, mask, rem, sc, sync);
    topk_emit<NT>(key, lo, hi, K, prefix, rem, out, sc, sync);
  }
  for (int j = K + tid; j < k_max; j += NT) out[j] = -1;
}

template <int NT, typename KeyFn>
__device__ __forceinline__ void topk_row(KeyFn key, int n, int K, int32_t *out, int k_max, TopkScratch<NT> &sc) {
  topk_row<NT>(key, n, K, out, k_max, sc, [] { __syncthreads(); });
}

// ---- Top-K of a row held in shared memory ---------------------------------------------------------
// The same selection as topk_row for a 512-thread block whose row of n <= 65535 keys sits in shared
// memory.  Thread tid owns the contiguous keys [tid C, tid C + C) (C from topk_chunk), so index order is
// thread order: each pass is independent work on a thread's own keys (16-byte loads) followed by one
// scan over the threads, instead of a ballot round per 32 keys (a shared load, a ballot and a
// count chained in every round).
//   1. Histogram of the keys' top 12 bits (4096 bins: the per-warp histograms; the caller may have
//      built it while making the keys, topk_h12_add) and the bin that holds the K-th largest key.
//   2. The keys of that bin are gathered into cand (any order).
//   3. Warp 0 narrows them to tau: one 8-bit pass (bits 19-12); the few keys left (at most 32)
//      rank themselves against each other across the lanes; else two more 8-bit passes.
//   4. Each thread counts its keys > tau and == tau (the keys above the bin, counted in step 2, and its
//      own gathered keys); a scan over the threads gives its first output slot and the keys == tau
//      before it, and it writes its kept indices: every key > tau and the keys == tau while fewer
//      than need_eq lie before (ties to the lower index, ascending output).
// A bin of more than kTopkCandCap keys (long runs of equal scores) takes three 8-bit block passes over
// the row instead of steps 2-3.  `stamp(k)` marks the end of phase k (0: histogram, 1: threshold bin,
// 2: tau, 3: indices written) for a diagnostic timeline; every thread calls it.
constexpr int kTopkCandCap = 1024;
constexpr int kTopkCand = kTopkCandCap + 32;  // cand entries: the gathered keys, then up to 32 left

// Adds key to the 4096-bin histogram of top-12-bit prefixes (zeroed TopkScratch<512>::hist).
__device__ __forceinline__ void topk_h12_add(uint32_t *h12, uint32_t key) { atomicAdd(&h12[key >> 20], 1u); }

// Keys per thread: a multiple of 4 (16-byte loads) that is 4 mod 8, so that the eight threads of a
// quarter-warp read eight distinct 4-bank groups.
__device__ __forceinline__ int topk_chunk(int n, int nt) {
  const int c = cdiv(n, nt);
  return c <= 4 ? 4 : 8 * cdiv(c - 4, 8) + 4;
}

// f(t, key) for t in [t0, t1) in index order; t0 a multiple of 4 and s_keys 16-byte aligned.
template <typename F>
__device__ __forceinline__ void topk_visit(const uint32_t *s_keys, int t0, int t1, F &&f) {
  int t = t0;
#pragma unroll 3
  for (; t + 4 <= t1; t += 4) {
    const uint4 q = *reinterpret_cast<const uint4 *>(s_keys + t);
    f(t, q.x);
    f(t + 1, q.y);
    f(t + 2, q.z);
    f(t + 3, q.w);
  }
  for (; t < t1; ++t) f(t, s_keys[t]);
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive scan of v over the block's NW warps in thread order, one barrier; s_warp must not be
// written again before a later barrier.
template <int NW>
__device__ __forceinline__ int block_excl_scan1(int v, int *s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int off = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) off += w < warp ? s_warp[w] : 0;
  return off + incl - v;
}

template <int NT, typename StampFn>
__device__ __forceinline__ void topk_row_smem(const uint32_t *s_keys, int n, int K, int32_t *out, int k_max,
                                              TopkScratch<NT> &sc, uint32_t *cand, bool hist_built, StampFn stamp) {
  static_assert(NT == 512, "4096 first-pass bins: the per-warp histograms of 16 warps, 8 per thread");
  constexpr int NW = NT / 32;
  auto sync = [] { __syncthreads(); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  if (K == n) {
    for (int t = tid; t < n; t += NT) out[t] = t;
  } else if (K > 0) {
    const int C = topk_chunk(n, NT);
    const int t0 = min(tid * C, n), t1 = min(t0 + C, n);
    uint32_t *h = &sc.hist[0][0];
    if (tid == 0) sc.ncand = 0;
    if (!hist_built) {
      for (int e = tid; e < NW * 256; e += NT) h[e] = 0u;
      sync();
      topk_visit(s_keys, t0, t1, [&](int, uint32_t k) { topk_h12_add(h, k); });
    }
    sync();
    stamp(0);
    // Thread tid owns bins 4095 - 8 tid .. 4088 - 8 tid (descending); the thread whose bins reach K
    // in the scan over the threads holds the threshold bin.
    uint32_t c[8];
    {
      const uint4 a = *reinterpret_cast<const uint4 *>(h + 4092 - 8 * tid);
      const uint4 b = *reinterpret_cast<const uint4 *>(h + 4088 - 8 * tid);
      c[0] = a.w; c[1] = a.z; c[2] = a.y; c[3] = a.x;
      c[4] = b.w; c[5] = b.z; c[6] = b.y; c[7] = b.x;
    }
    int sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += (int)c[j];
    const int excl = block_excl_scan1<NW>(sum, sc.wgt);
    if (excl < K && excl + sum >= K) {
      int run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run + (int)c[j] >= K) {
          sc.digit = 4095u - 8u * tid - j;
          sc.rem = K - run;
          sc.cbin = (int)c[j];
          break;
        }
        run += (int)c[j];
      }
    }
    sync();
    stamp(1);
    uint32_t prefix = sc.digit << 20, mask = 0xfff00000u;
    int rem = sc.rem;
    const int nb = sc.cbin;
    uint32_t tau;
    int need_eq;
    int gt_pre = -1, cand_mine = 0, cand_cnt = 0;  // gathered path: keys above the bin, own gathered keys
    if (nb <= kTopkCandCap) {
      int cin = 0, above = 0;
      topk_visit(s_keys, t0, t1, [&](int, uint32_t k) {
        const uint32_t top = k & mask;
        cin += top == prefix ? 1 : 0;
        above += top > prefix ? 1 : 0;
      });
      const int incl = warp_incl_scan(cin);
      int base = 0;
      if (lane == 31 && incl > 0) base = atomicAdd(&sc.ncand, incl);
      base = __shfl_sync(0xffffffffu, base, 31) + incl - cin;
      const int mine = base;  // this thread's gathered keys are cand[mine, mine + cin)
      if (cin > 0)
        topk_visit(s_keys, t0, t1, [&](int, uint32_t k) {
          if ((k & mask) == prefix) cand[base++] = k;
        });
      gt_pre = above;
      cand_mine = mine;
      cand_cnt = cin;
      sync();
      if (warp == 0) {
        uint32_t *hw = sc.tot;
#pragma unroll
        for (int e = lane; e < 256; e += 32) hw[e] = 0u;
        __syncwarp();
        for (int i = lane; i < nb; i += 32) atomicAdd(&hw[(cand[i] >> 12) & 255u], 1u);
        __syncwarp();
        uint32_t d;
        warp_find_digit(hw, rem, d, rem);
        prefix |= d << 12;
        mask |= 0xffu << 12;
        // The keys left (their top 20 bits are prefix), compacted after the gathered ones.
        uint32_t *left = cand + kTopkCandCap;
        int m = 0;
        for (int i0 = 0; i0 < nb; i0 += 32) {
          const int i = i0 + lane;
          const uint32_t k = i < nb ? cand[i] : 0u;
          const bool in = i < nb && (k & mask) == prefix;
          const unsigned bm = __ballot_sync(0xffffffffu, in);
          const int j = m + __popc(bm & lt);
          if (in && j < 32) left[j] = k;
          m += __popc(bm);
        }
        __syncwarp();
        if (m <= 32) {
          // tau is the rem-th largest of the m keys left: the key with fewer than rem keys above it
          // and at least rem at or above it.
          const bool have = lane < m;
          const uint32_t v = have ? left[lane] : 0u;
          int gt = 0, ge = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t vj = __shfl_sync(0xffffffffu, v, j);
            const int in = j < m ? 1 : 0;
            gt += (vj > v ? 1 : 0) & in;
            ge += (vj >= v ? 1 : 0) & in;
          }
          const int f = __ffs(__ballot_sync(0xffffffffu, have && gt < rem && rem <= ge)) - 1;
          tau = __shfl_sync(0xffffffffu, v, f);
          need_eq = rem - __shfl_sync(0xffffffffu, gt, f);
        } else {
#pragma unroll 1
          for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 4 : 0;
#pragma unroll
            for (int e = lane; e < 256; e += 32) hw[e] = 0u;
            __syncwarp();
            for (int i = lane; i < nb; i += 32) {
              const uint32_t k = cand[i];
              if ((k & mask) == prefix) atomicAdd(&hw[(k >> shift) & 255u], 1u);
            }
            __syncwarp();
            warp_find_digit(hw, rem, d, rem);
            prefix |= d << shift;
            mask |= 0xffu << shift;
            __syncwarp();
          }
          tau = prefix;
          need_eq = rem;
        }
        if (lane == 0) {
          sc.digit = tau;
          sc.rem = need_eq;
        }
      }
      sync();
      tau = sc.digit;
      need_eq = sc.rem;
    } else {
      // Warp-range passes (topk_block_pass) over the whole row.
      const int seg = cdiv(cdiv(n, NW), 32) * 32;
      const int lo = min(warp * seg, n), hi = min(lo + seg, n);
      auto key = [&](int t) -> uint32_t { return s_keys[t]; };
      for (int e = tid; e < NW * 256; e += NT) h[e] = 0u;
      sync();
      topk_block_pass<NT>(key, lo, hi, 12, prefix, mask, rem, sc, sync);
      topk_block_pass<NT>(key, lo, hi, 4, prefix, mask, rem, sc, sync);
      topk_block_pass<NT>(key, lo, hi, 0, prefix, mask, rem, sc, sync);
      tau = prefix;
      need_eq = rem;
    }
    stamp(2);
    int gt = 0, eq = 0;
    if (gt_pre >= 0) {
      // Keys above the threshold bin are all > tau; of the bin's keys only this thread's own decide.
      gt = gt_pre;
      for (int i = 0; i < cand_cnt; ++i) {
        const uint32_t k = cand[cand_mine + i];
        gt += k > tau ? 1 : 0;
        eq += k == tau ? 1 : 0;
      }
    } else {
      topk_visit(s_keys, t0, t1, [&](int, uint32_t k) {
        gt += k > tau ? 1 : 0;
        eq += k == tau ? 1 : 0;
      });
    }
    // Both counts in one scan (each total is at most n < 2^16).
    const int pk = block_excl_scan1<NW>(gt | eq << 16, sc.weq);
    const int pgt = pk & 0xffff, peq = pk >> 16;
    int pos = pgt + min(peq, need_eq), run_eq = peq;
    topk_visit(s_keys, t0, t1, [&](int t, uint32_t k) {
      const bool e = k == tau;
      if (k > tau || (e && run_eq < need_eq)) {
        if (pos < K) out[pos] = t;
        ++pos;
      }
      run_eq += e ? 1 : 0;
    });
  }
  for (int j = K + tid; j < k_max; j += NT) out[j] = -1;
  stamp(3);
}

template <int NT>
__device__ __forceinline__ void topk_row_smem(const uint32_t *s_keys, int n, int K, int32_t *out, int k_max,
                                              TopkScratch<NT> &sc, uint32_t *cand, bool hist_built) {
  topk_row_smem<NT>(s_keys, n, K, out, k_max, sc, cand, hist_built, [](int) {});
}

}  // namespace ssd
