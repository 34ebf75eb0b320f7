// ssd_select.cu -- Top-K selection of critical tokens (or blocks) and the union of the candidates'
// block sets.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: Top-K over the dumped, GQA-reduced verify scores gives the sparse
// pattern; §3.2 / §5.4: about 5% of the tokens.  SpecSA post, overlap-aware grouped query execution
// and the hierarchical layout representation: the candidates' block sets are merged into one
// ordered union with a per-block candidate mask.
//
// One block selects one row with topk_row_smem (a row staged in shared memory) or topk_row (a longer
// row read from global memory); ssd_topk.cuh: exact radix select, ties to the lower index, output
// sorted.
#include "ssd_host.h"
#include "ssd_topk.cuh"

namespace ssd {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelTile = kSelThreads * kSelItems;
constexpr int kSelSmemRow = 40960;  // rows up to this length are staged in shared memory

struct TopkArgs {
  const float *scores;
  int64_t stride;
  const int32_t *lens;
  const int32_t *ks;
  int rows_per_group, len_div, max_len;
  int32_t *idx;
  int k_max;
  int32_t *cnt;
  unsigned *status;
  int ks_per_row;  // ks indexed by row (top-p counts) instead of by group
};

template <bool IN_SMEM>
__global__ void __launch_bounds__(kSelThreads) topk_kernel(TopkArgs p) {
  extern __shared__ uint32_t s_keys[];
  __shared__ TopkScratch<kSelThreads> sc;
  __shared__ uint32_t s_cand[kTopkCand];
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int grp = (int)(row / p.rows_per_group);
  pdl_wait();
  int raw_len = p.lens[grp];
  int n = raw_len <= 0 ? 0 : cdiv(raw_len, p.len_div);
  if (raw_len < 0 || n > p.max_len) {
    if (tid == 0) atomicOr(p.status, (unsigned)SSD_FAULT_SEQLEN);
    n = n > p.max_len ? p.max_len : n;
  }
  int K = p.ks_per_row ? p.ks[row] : p.ks[grp];
  K = K < 0 ? 0 : (K > n ? n : K);
  if (K > p.k_max) {
    if (tid == 0) atomicOr(p.status, (unsigned)SSD_FAULT_KMAX);
    K = p.k_max;
  }
  const float *src = p.scores + row * p.stride;
  int32_t *out = p.idx + row * p.k_max;
  if (IN_SMEM) {
    // The keys, and the histogram of their top 12 bits that the selection starts from.
    for (int e = tid; e < kSelWarps * 256; e += kSelThreads) (&sc.hist[0][0])[e] = 0u;
    __syncthreads();
    for (int t = tid; t < n; t += kSelThreads) {
      const uint32_t k = score_key(src[t]);
      s_keys[t] = k;
      topk_h12_add(&sc.hist[0][0], k);
    }
    __syncthreads();
  }
  auto key = [&](int t) -> uint32_t { return IN_SMEM ? s_keys[t] : score_key(__ldg(src + t)); };

  pdl_trigger();
  if (IN_SMEM)
    topk_row_smem<kSelThreads>(s_keys, n, K, out, p.k_max, sc, s_cand, true);
  else
    topk_row<kSelThreads>(key, n, K, out, p.k_max, sc);
  if (tid == 0) p.cnt[row] = K;
}

// Top-p counts: K_p(row) = the smallest number of the row's largest entries (ties toward the lower
// index) whose sum reaches p times the row total, capped at k_max.  Sums are taken in 64-bit fixed
// point, exactly and in any order: with E the largest biased exponent in the row, each value
// m * 2^(E' - 150) (m its 24-bit significand) becomes floor(value * 2^(188 - E - ceil(log2 n))), so
// the row total stays below 2^62; values below 2^(ceil(log2 n) - 62) times the row maximum round
// down.  target = ceil(p * total).  The search is the radix select above run on bucket sums as well
// as counts: each 8-bit pass walks the buckets from the highest digit down, adds whole buckets while
// the running sum stays below the target and descends into the bucket where it is reached; the
// entries equal to the final key tau (one value) are then counted in closed form.  The kept set is
// the Top-K set of the row with K = K_p, so the indices come from topk_kernel.
struct ToppArgs {
  const float *scores;
  int64_t stride;
  const int32_t *lens;
  double p;
  int rows_per_group, len_div, max_len, k_max;
  int32_t *k_rows;
  unsigned *status;
};

// Fixed-point value of a non-negative score key: floor(value * 2^(shift0 + 150 - 1)) with the
// exponent offset folded into shift0 (= e - 149 for the row's scale 2^e).
__device__ __forceinline__ uint64_t key_fixed(uint32_t k, int shift0) {
  const uint32_t u = k & 0x7fffffffu;  // keys of non-negative values carry the top bit
  int E = (int)(u >> 23);
  uint32_t m = u & 0x7fffffu;
  if (E) m |= 0x800000u; else E = 1;
  const int sh = E + shift0;  // value * 2^e = m * 2^(E - 150 + e)
  if (sh >= 0) return (uint64_t)m << sh;
  return -sh >= 24 ? 0ull : (uint64_t)(m >> -sh);
}

template <bool IN_SMEM>
__global__ void __launch_bounds__(kSelThreads) topp_k_kernel(ToppArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ uint32_t s_hist[kSelWarps][256];
  __shared__ unsigned long long s_qsum[kSelWarps][256];
  __shared__ uint32_t s_tot[256];
  __shared__ uint64_t s_tsum[256];
  __shared__ uint32_t s_digit, s_kmax;
  __shared__ uint64_t s_above, s_target;
  __shared__ int s_above_n, s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int grp = (int)(row / a.rows_per_group);
  pdl_trigger();
  pdl_wait();
  const int raw_len = a.lens[grp];
  int n = raw_len <= 0 ? 0 : cdiv(raw_len, a.len_div);
  if (raw_len < 0 || n > a.max_len) {
    if (tid == 0) atomicOr(a.status, (unsigned)SSD_FAULT_SEQLEN);
    n = n > a.max_len ? a.max_len : n;
  }
  const float *src = a.scores + row * a.stride;
  if (tid == 0) {
    s_bad = 0;
    s_kmax = 0u;
  }
  __syncthreads();
  int bad = 0;
  uint32_t kmax = 0u;
  for (int t = tid; t < n; t += kSelThreads) {
    const float v = src[t];
    bad |= !(v >= 0.f);  // negative or NaN
    const uint32_t k = score_key(v);
    kmax = k > kmax ? k : kmax;
    if (IN_SMEM) s_keys[t] = k;
  }
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) atomicMax(&s_kmax, kmax);
  if (bad) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      atomicOr(a.status, (unsigned)SSD_FAULT_VALUE);
      a.k_rows[row] = 0;
    }
    return;
  }
  // An all-zero (or empty) row, or p = 0, keeps nothing: the target is 0.
  if (n == 0 || !(a.p > 0.0) || (s_kmax & 0x7fffffffu) == 0u) {
    if (tid == 0) a.k_rows[row] = 0;
    return;
  }
  const int Emax = max((int)((s_kmax & 0x7fffffffu) >> 23), 1);
  const int lg = n > 1 ? 32 - __clz(n - 1) : 0;
  const int shift0 = (188 - Emax - lg) - 150;
  auto key = [&](int t) -> uint32_t { return IN_SMEM ? s_keys[t] : score_key(__ldg(src + t)); };
  uint32_t prefix = 0, mask = 0;
  uint64_t above = 0;  // fixed-point sum of the entries known to be kept (keys above the path)
  int above_n = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int e = tid; e < kSelWarps * 256; e += kSelThreads) {
      (&s_hist[0][0])[e] = 0u;
      (&s_qsum[0][0])[e] = 0ull;
    }
    __syncthreads();
    for (int t = tid; t < n; t += kSelThreads) {
      const uint32_t k = key(t);
      if ((k & mask) == prefix) {
        const uint32_t dg = (k >> shift) & 255u;
        atomicAdd(&s_hist[warp][dg], 1u);
        atomicAdd(&s_qsum[warp][dg], (unsigned long long)key_fixed(k, shift0));
      }
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t c = 0;
      uint64_t q = 0;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) {
        c += s_hist[w][tid];
        q += s_qsum[w][tid];
      }
      s_tot[tid] = c;
      s_tsum[tid] = q;
    }
    __syncthreads();
    if (warp == 0) {
      // Lane l owns digits 255-8l .. 248-8l (descending).
      uint32_t c[8];
      uint64_t q[8];
      uint64_t lsum = 0;
      int lcnt = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = s_tot[255 - 8 * lane - j];
        q[j] = s_tsum[255 - 8 * lane - j];
        lsum += q[j];
        lcnt += (int)c[j];
      }
      uint64_t incl = lsum;
      int incl_n = lcnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        const int tn = __shfl_up_sync(0xffffffffu, incl_n, o);
        if (lane >= o) {
          incl += t;
          incl_n += tn;
        }
      }
      if (pass == 0 && lane == 31) {
        // incl is now the exact row total (< 2^62).
        const double tg = ceil(a.p * (double)incl);
        s_target = tg >= (double)incl ? incl : (uint64_t)tg;
      }
      __syncwarp();
      const uint64_t target = s_target;
      // Entries above this lane's digits are kept: the first digit whose bucket reaches the
      // target is the one to descend into (a bucket holds at least one entry; the last
      // non-empty digit is reached at the latest, as the buckets sum to what remains).
      const uint64_t excl = incl - lsum;
      const int excl_n = incl_n - lcnt;
      uint64_t run = above + excl;
      int run_n = above_n + excl_n, hit = -1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (hit < 0 && c[j] != 0u) {
          if (run + q[j] >= target)
            hit = j;
          else {
            run += q[j];
            run_n += (int)c[j];
          }
        }
      }
      const unsigned hits = __ballot_sync(0xffffffffu, hit >= 0);
      if (lane == __ffs(hits) - 1) {
        s_digit = 255u - 8u * lane - (unsigned)hit;
        s_above = run;
        s_above_n = run_n;
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 0xffu << shift;
    above = s_above;
    above_n = s_above_n;
    __syncthreads();
  }
  if (tid == 0) {
    // Entries equal to tau: the smallest m with above + m * v >= target (v > 0 here, or the
    // bucket would not have been reached), capped by how many there are.
    const uint64_t v = key_fixed(prefix, shift0), need = s_target - above;
    const int eq = (int)s_tot[prefix & 255u];
    uint64_t m = v ? (need + v - 1) / v : (uint64_t)eq;
    if (m > (uint64_t)eq) m = (uint64_t)eq;
    const int K = above_n + (int)m;
    a.k_rows[row] = K < a.k_max ? K : a.k_max;
  }
}

// Union of block sets: one block per unit; a shared bitmap holds each block's candidate mask.
struct UnionArgs {
  const int32_t *blocks;
  const int32_t *bcnt;
  int n_c, kb, nblk_max;
  int32_t *uidx;
  uint32_t *umask;
  int32_t *ucnt;
  int umax;
  unsigned *status;
};

__global__ void __launch_bounds__(kSelThreads) union_kernel(UnionArgs p) {
  extern __shared__ uint32_t s_mask[];
  __shared__ int s_warp[kSelWarps];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int64_t u = blockIdx.x;
  pdl_trigger();
  for (int j = tid; j < p.nblk_max; j += kSelThreads) s_mask[j] = 0u;
  pdl_wait();
  __syncthreads();
  for (int e = tid; e < p.n_c * p.kb; e += kSelThreads) {
    int i = e / p.kb, j = e % p.kb;
    int c = p.bcnt[u * p.n_c + i];
    c = c < 0 ? 0 : (c > p.kb ? p.kb : c);
    if (j < c) {
      int blk = p.blocks[(u * p.n_c + i) * p.kb + j];
      if (blk >= 0 && blk < p.nblk_max) atomicOr(&s_mask[blk], 1u << i);
      else atomicOr(p.status, (unsigned)SSD_FAULT_INDEX);
    }
  }
  __syncthreads();
  int base = 0;
  for (int start = 0; start < p.nblk_max; start += kSelTile) {
    const int j0 = start + tid * kSelItems;
    int c = 0;
#pragma unroll
    for (int e = 0; e < kSelItems; ++e) c += (j0 + e < p.nblk_max && s_mask[j0 + e]) ? 1 : 0;
    int pos = base + block_excl_scan<kSelWarps>(c, s_warp, &s_total);
    const int tot = s_total;
#pragma unroll
    for (int e = 0; e < kSelItems; ++e) {
      int j = j0 + e;
      if (j < p.nblk_max && s_mask[j]) {
        if (pos < p.umax) {
          p.uidx[u * p.umax + pos] = j;
          p.umask[u * p.umax + pos] = s_mask[j];
        } else {
          atomicOr(p.status, (unsigned)SSD_FAULT_UNION);
        }
        ++pos;
      }
    }
    base += tot;
  }
  const int n = base < p.umax ? base : p.umax;
  for (int j = n + tid; j < p.umax; j += kSelThreads) {
    p.uidx[u * p.umax + j] = -1;
    p.umask[u * p.umax + j] = 0u;
  }
  if (tid == 0) p.ucnt[u] = n;
}

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_select_topk(const float *scores, int64_t stride, const int32_t *lens, const int32_t *ks,
                               int n_groups, int rows_per_group, int len_div, int max_len, int32_t *idx, int k_max,
                               int32_t *cnt, ssd_stream_t stream) {
  const char *who = "ssd_select_topk";
  if (!scores || !lens || !ks || !cnt || (!idx && k_max > 0))
    return fail(SSD_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (n_groups < 0 || rows_per_group <= 0 || len_div <= 0 || max_len < 0 || k_max < 0)
    return fail(SSD_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (stride < max_len) return fail(SSD_ERR_INVALID_ARG, "%s: stride %lld < max_len %d", who, (long long)stride, max_len);
  const int64_t rows = (int64_t)n_groups * rows_per_group;
  if (rows == 0) return SSD_OK;
  if (rows > (1ll << 31) - 1) return fail(SSD_ERR_UNSUPPORTED, "%s: too many rows", who);
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  TopkArgs p{scores, stride, lens, ks, rows_per_group, len_div, max_len, idx, k_max, cnt, status, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (max_len <= kSelSmemRow) {
    const int smem = (max_len > 0 ? max_len : 1) * 4;
    int rc = ensure_smem<topk_kernel<true>>(smem);
    if (rc) return rc;
    return launch(topk_kernel<true>, dim3((unsigned)rows), dim3(kSelThreads), smem, st, "topk_kernel", p);
  }
  return launch(topk_kernel<false>, dim3((unsigned)rows), dim3(kSelThreads), 0, st, "topk_kernel", p);
}

extern "C" int ssd_block_union(const int32_t *blocks, const int32_t *bcnt, int n_units, int n_cand, int kb,
                               int nblk_max, int32_t *uidx, uint32_t *umask, int32_t *ucnt, int umax,
                               ssd_stream_t stream) {
  const char *who = "ssd_block_union";
  if (!blocks || !bcnt || !uidx || !umask || !ucnt) return fail(SSD_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (n_units < 0 || n_cand < 1 || kb < 0 || nblk_max < 1 || umax < 1)
    return fail(SSD_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (n_cand > 32) return fail(SSD_ERR_UNSUPPORTED, "%s: n_cand %d > 32", who, n_cand);
  if (nblk_max > kSelSmemRow) return fail(SSD_ERR_UNSUPPORTED, "%s: nblk_max %d > %d", who, nblk_max, kSelSmemRow);
  if (n_units == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  UnionArgs p{blocks, bcnt, n_cand, kb, nblk_max, uidx, umask, ucnt, umax, status};
  const int smem = nblk_max * 4;
  int rc = ensure_smem<union_kernel>(smem);
  if (rc) return rc;
  return launch(union_kernel, dim3(n_units), dim3(kSelThreads), smem, reinterpret_cast<cudaStream_t>(stream),
                "union_kernel", p);
}

extern "C" int ssd_select_topp(const float *scores, int64_t stride, const int32_t *lens, float p, int n_groups,
                               int rows_per_group, int len_div, int max_len, int32_t *idx, int k_max, int32_t *cnt,
                               int32_t *k_rows, ssd_stream_t stream) {
  const char *who = "ssd_select_topp";
  if (!scores || !lens || !cnt || !k_rows || (!idx && k_max > 0)) return fail(SSD_ERR_INVALID_ARG, "%s: NULL pointer", who);
  if (!(p >= 0.f && p <= 1.f)) return fail(SSD_ERR_INVALID_ARG, "%s: p must be in [0, 1]", who);
  if (n_groups < 0 || rows_per_group <= 0 || len_div <= 0 || max_len < 0 || k_max < 0)
    return fail(SSD_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (stride < max_len) return fail(SSD_ERR_INVALID_ARG, "%s: stride %lld < max_len %d", who, (long long)stride, max_len);
  const int64_t rows = (int64_t)n_groups * rows_per_group;
  if (rows == 0) return SSD_OK;
  if (rows > (1ll << 31) - 1) return fail(SSD_ERR_UNSUPPORTED, "%s: too many rows", who);
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ToppArgs ta{scores, stride, lens, (double)p, rows_per_group, len_div, max_len, k_max, k_rows, status};
  TopkArgs tk{scores, stride, lens, k_rows, rows_per_group, len_div, max_len, idx, k_max, cnt, status, 1};
  if (max_len <= kSelSmemRow) {
    const int smem = (max_len > 0 ? max_len : 1) * 4;
    int rc = ensure_smem<topp_k_kernel<true>>(smem);
    if (rc) return rc;
    if ((rc = ensure_smem<topk_kernel<true>>(smem))) return rc;
    if ((rc = launch(topp_k_kernel<true>, dim3((unsigned)rows), dim3(kSelThreads), smem, st, "topp_k_kernel", ta)))
      return rc;
    return launch(topk_kernel<true>, dim3((unsigned)rows), dim3(kSelThreads), smem, st, "topk_kernel", tk);
  }
  int rc = launch(topp_k_kernel<false>, dim3((unsigned)rows), dim3(kSelThreads), 0, st, "topp_k_kernel", ta);
  if (rc) return rc;
  return launch(topk_kernel<false>, dim3((unsigned)rows), dim3(kSelThreads), 0, st, "topk_kernel", tk);
}
