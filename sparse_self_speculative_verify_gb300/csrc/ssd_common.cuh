// ssd_common.cuh -- device helpers shared by the libssd kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// Verify work item: a split of kSplitTokens consecutive tokens of one (request, KV head).
constexpr int kSplitTokens = 512;
// Split length of the fp32 (CUDA-core) verify: shorter, so that small batches still spread over
// many blocks.
constexpr int kSimtSplitTokens = 128;
// Tokens staged in shared memory per pipeline step of the verify kernels.
constexpr int kStageTokens = 64;
// Criticality side values carry one log2-domain reference per (row, kRefGroup tokens).
constexpr int kRefGroup = 16;
constexpr int kRefShift = 4;    // log2(kRefGroup): one reference per 16 tokens (the mma.sync and SIMT verify)
constexpr int kTcRefShift = 7;  // the tensor-core verify: one reference per 128-token tile
// Row stride of the per-row references with one reference per (1 << ref_shift) tokens: a multiple of
// four floats, so that every row starts 16-byte aligned (Lpad / 16 already is one).
__host__ __device__ constexpr int ref_stride(int Lpad, int ref_shift) { return ((Lpad >> ref_shift) + 3) / 4 * 4; }
// Row length of the criticality side buffer is a multiple of this (the largest tile that writes it).
constexpr int kSideAlign = 128;
// Draft work item: up to kDraftChunk selected tokens of one (request, KV head).
constexpr int kDraftChunk = 64;
// Tokens per union block in the block-granular path.
constexpr int kBlockTokens = 64;
// Union blocks per block-sparse work item.
constexpr int kBlocksPerItem = 8;
constexpr int kMaxRows = 64;  // R = G * n_cand
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Paged cache as the kernels see it.
struct KVView {
  const void *pool;
  int64_t num_pages;
  int page_size;
  int log2_ps;
  int h_kv;
  const int32_t *page_table;
  int max_pages;
  const int32_t *seq_lens;
  int batch;
  int max_seq_len;
};

// Effective length of request b: clamped to what the page table and grid can hold; a value
// outside [lo, max] raises SSD_FAULT_SEQLEN.
__device__ __forceinline__ int effective_len(const KVView &kv, int b, int lo, unsigned *status) {
  int L = kv.seq_lens[b];
  int hi = kv.max_seq_len;
  if (L < lo || L > hi) {
    atomicOr(status, (unsigned)SSD_FAULT_SEQLEN);
    L = L < 0 ? 0 : (L > hi ? hi : L);
  }
  return L;
}

// Byte address of row (K or V, head g, token t) of request b; nullptr (and SSD_FAULT_PAGE) when
// the page id is outside the pool.
template <int D, typename T>
__device__ __forceinline__ const T *kv_row(const KVView &kv, int b, int which, int g, int t,
                                           unsigned *status) {
  int j = t >> kv.log2_ps;
  int32_t p = __ldg(kv.page_table + (int64_t)b * kv.max_pages + j);
  if (p < 0 || (int64_t)p >= kv.num_pages) {
    atomicOr(status, (unsigned)SSD_FAULT_PAGE);
    return nullptr;
  }
  int64_t row = (((int64_t)p * 2 + which) * kv.h_kv + g) * kv.page_size + (t & (kv.page_size - 1));
  return reinterpret_cast<const T *>(kv.pool) + row * D;
}

// Programmatic dependent launch.  Every kernel of the library is launched so that it may start
// while the kernel before it on the stream is finishing: its blocks can be placed on SMs the earlier
// grid has left and run work that reads nothing an earlier kernel wrote (shared-memory and barrier
// set-up, tensor-memory allocation).  pdl_wait() returns once every grid this one depends on has
// completed and its memory is visible; each kernel calls it in every block before its first access
// to global memory that an earlier kernel may write (and before it exits), so the completion of any
// kernel implies the completion of all kernels before it on the stream.  Without the launch
// attribute both instructions do nothing.  pdl_trigger() lets the next kernel's launch begin once
// every block of this grid has issued it (or exited); kernels issue it when a block's remaining
// work is short (its last item, stage or chunk), so the next kernel's blocks arrive during this
// one's tail rather than sitting on SMs through all of it (issued at kernel entry it measured
// slower than no dependent launch at all).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// L2 policy that keeps lines in L2 ahead of normal and evict-first ones.
__device__ __forceinline__ uint64_t policy_l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte global store under an L2 cache policy.
__device__ __forceinline__ void st_global_policy(void *dst, const uint4 &v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}
// Drops the 128-byte L2 line at `p` (128-byte aligned) without writing it back to memory; its contents
// become undefined.  For scratch data that has been read for the last time.
__device__ __forceinline__ void discard_l2_line(const void *p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// 16-byte asynchronous global->shared copy; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x via the hardware approximation (max relative error about 2^-22); ex2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_half(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Split a pair of fp32 values into bf16 high parts and bf16 residuals: v ~= hi + lo with a
// relative error of about 2^-16, so a probability carried through two bf16 MMAs keeps ~16 bits.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t &hi, uint32_t &lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = pack_bf16(a - hf.x, b - hf.y);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Element offset of (row, 16-byte chunk c) in a tile whose rows hold `cpr` 16-byte chunks, with
// the chunk index XOR-swizzled by the row so that 8 consecutive rows of one logical chunk fall in
// 8 different bank groups.
__device__ __forceinline__ int swz_chunk(int row, int c) { return c ^ (row & 7); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace ssd
