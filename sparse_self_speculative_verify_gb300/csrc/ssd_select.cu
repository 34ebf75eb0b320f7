// ssd_select.cu -- Top-K selection of critical tokens (or blocks) and the union of the candidates'
// block sets.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: Top-K over the dumped, GQA-reduced verify scores gives the sparse
// pattern; §3.2 / §5.4: about 5% of the tokens.  SpecSA post, overlap-aware grouped query execution
// and the hierarchical layout representation: the candidates' block sets are merged into one
// ordered union with a per-block candidate mask.
//
// Selection is an exact radix select on the order-preserving 32-bit key of each fp32 score (four
// 8-bit MSB-first histogram passes find the K-th largest key tau), followed by a stream compaction
// in index order that keeps every key > tau and the lowest-index keys == tau until K are kept, so
// ties go to the lower index and the output comes out sorted.
#include "ssd_host.h"

namespace ssd {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelItems = 4;
constexpr int kSelTile = kSelThreads * kSelItems;
constexpr int kSelSmemRow = 40960;  // rows up to this length are staged in shared memory

// Order-preserving key: unsigned order of the keys = numeric order of the floats; -0.0 == +0.0.
__device__ __forceinline__ uint32_t score_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one value per thread; *total receives the sum.
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
    int w = lane < kSelWarps ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kSelWarps) s_warp[lane] = wi - w;
    if (lane == kSelWarps - 1) *s_total = wi;
  }
  __syncthreads();
  int res = s_warp[warp] + incl - v;
  __syncthreads();
  return res;
}

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
};

template <bool IN_SMEM>
__global__ void __launch_bounds__(kSelThreads) topk_kernel(TopkArgs p) {
  extern __shared__ uint32_t s_keys[];
  __shared__ uint32_t s_hist[kSelWarps][256];
  __shared__ uint32_t s_tot[256];
  __shared__ int s_warp[kSelWarps];
  __shared__ int s_total;
  __shared__ uint32_t s_digit;
  __shared__ int s_rem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int grp = (int)(row / p.rows_per_group);
  int raw_len = p.lens[grp];
  int n = raw_len <= 0 ? 0 : cdiv(raw_len, p.len_div);
  if (raw_len < 0 || n > p.max_len) {
    if (tid == 0) atomicOr(p.status, (unsigned)SSD_FAULT_SEQLEN);
    n = n > p.max_len ? p.max_len : n;
  }
  int K = p.ks[grp];
  K = K < 0 ? 0 : (K > n ? n : K);
  if (K > p.k_max) {
    if (tid == 0) atomicOr(p.status, (unsigned)SSD_FAULT_KMAX);
    K = p.k_max;
  }
  const float *src = p.scores + row * p.stride;
  int32_t *out = p.idx + row * p.k_max;
  if (IN_SMEM) {
    for (int t = tid; t < n; t += kSelThreads) s_keys[t] = score_key(src[t]);
    __syncthreads();
  }
  auto key = [&](int t) -> uint32_t { return IN_SMEM ? s_keys[t] : score_key(__ldg(src + t)); };

  if (K == n) {
    for (int t = tid; t < n; t += kSelThreads) out[t] = t;
  } else if (K > 0) {
    uint32_t prefix = 0, mask = 0;
    int rem = K;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int e = tid; e < kSelWarps * 256; e += kSelThreads) (&s_hist[0][0])[e] = 0u;
      __syncthreads();
      for (int t = tid; t < n; t += kSelThreads) {
        uint32_t k = key(t);
        if ((k & mask) == prefix) atomicAdd(&s_hist[warp][(k >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 256) {
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kSelWarps; ++w) s += s_hist[w][tid];
        s_tot[tid] = s;
      }
      __syncthreads();
      if (warp == 0) {
        // Lane l owns bins 255-8l .. 248-8l (descending).
        uint32_t c[8];
        uint32_t sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s_tot[255 - 8 * lane - j];
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
              s_digit = 255u - 8u * lane - j;
              s_rem = rem - (int)run;
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= 0xffu << shift;
      rem = s_rem;
      __syncthreads();
    }
    const uint32_t tau = prefix;
    const int need_eq = rem;
    int base_eq = 0, base_sel = 0;
    for (int start = 0; start < n; start += kSelTile) {
      const int t_first = start + tid * kSelItems;
      uint32_t kk[kSelItems];
      int c_eq = 0;
#pragma unroll
      for (int e = 0; e < kSelItems; ++e) {
        int t = t_first + e;
        kk[e] = t < n ? key(t) : 0u;
        c_eq += (t < n && kk[e] == tau) ? 1 : 0;
      }
      const int ex_eq = block_excl_scan(c_eq, s_warp, &s_total);
      const int tot_eq = s_total;
      int run = base_eq + ex_eq;
      unsigned sel = 0;
#pragma unroll
      for (int e = 0; e < kSelItems; ++e) {
        int t = t_first + e;
        if (t < n) {
          if (kk[e] == tau) {
            if (run < need_eq) sel |= 1u << e;
            ++run;
          } else if (kk[e] > tau) {
            sel |= 1u << e;
          }
        }
      }
      const int ex_sel = block_excl_scan(__popc(sel), s_warp, &s_total);
      const int tot_sel = s_total;
      int pos = base_sel + ex_sel;
#pragma unroll
      for (int e = 0; e < kSelItems; ++e)
        if ((sel >> e) & 1u) {
          if (pos < K) out[pos] = t_first + e;
          ++pos;
        }
      base_eq += tot_eq;
      base_sel += tot_sel;
    }
  }
  for (int j = K + tid; j < p.k_max; j += kSelThreads) out[j] = -1;
  if (tid == 0) p.cnt[row] = K;
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
  for (int j = tid; j < p.nblk_max; j += kSelThreads) s_mask[j] = 0u;
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
    int pos = base + block_excl_scan(c, s_warp, &s_total);
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
  TopkArgs p{scores, stride, lens, ks, rows_per_group, len_div, max_len, idx, k_max, cnt, status};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (max_len <= kSelSmemRow) {
    const int smem = (max_len > 0 ? max_len : 1) * 4;
    int rc = ensure_smem<topk_kernel<true>>(smem);
    if (rc) return rc;
    topk_kernel<true><<<(unsigned)rows, kSelThreads, smem, st>>>(p);
  } else {
    topk_kernel<false><<<(unsigned)rows, kSelThreads, 0, st>>>(p);
  }
  return check_launch("topk_kernel");
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
  union_kernel<<<n_units, kSelThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return check_launch("union_kernel");
}
