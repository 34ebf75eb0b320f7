// ssd_kv.cu -- KV append into the paged cache and sequence-length advance (accept / reject).
//
// SpecSA ("SpecSA：融合推测解码与稀疏注意力的高效LLM推理框架"), "refresh/reuse NSA kernel fusion" and
// "branch handling": the KV of accepted tokens stays for later queries, that of rejected tokens is
// dropped.  SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative
// Decoding with Sparse Attention") §2.3: a verify checks the k drafted tokens plus one bonus position.
// With the verify convention of this library (a request's n_c candidates occupy its last n_c
// positions), a round is: append the candidates' K/V at seq_lens[b] .. seq_lens[b] + n_c - 1, advance
// the lengths by n_c, verify, then advance by -(n_c - accepted_b): the rejected candidates' rows stay
// in their pages but lie past the request's end, where no kernel reads them.
#include "ssd_host.h"

namespace ssd {

constexpr int kAppendThreads = 256;

// One block per request.  The request is skipped (and flagged) when any of its new positions would
// pass max_seq_len or fall in a page id outside the pool, so a request is either fully appended or
// untouched.  Rows move as 16-byte pieces: a piece is (token j, KV head g, K|V, 16-byte chunk c).
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(KVView kv, char *pool, const char *k_new,
                                                                   const char *v_new, int n_new, int row_bytes,
                                                                   unsigned *status) {
  const int b = blockIdx.x, tid = threadIdx.x;
  __shared__ int s_ok;
  pdl_trigger();
  pdl_wait();
  const int L = kv.seq_lens[b];
  if (tid == 0) s_ok = 1;
  __syncthreads();
  const bool len_ok = L >= 0 && (int64_t)L + n_new <= kv.max_seq_len;
  if (!len_ok) {
    if (tid == 0) atomicOr(status, (unsigned)SSD_FAULT_SEQLEN);
    return;
  }
  // Every page the new tokens touch must exist.
  for (int j = tid; j < n_new; j += kAppendThreads) {
    const int32_t p = kv.page_table[(int64_t)b * kv.max_pages + ((L + j) >> kv.log2_ps)];
    if (p < 0 || (int64_t)p >= kv.num_pages) s_ok = 0;
  }
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) atomicOr(status, (unsigned)SSD_FAULT_PAGE);
    return;
  }
  const int cpr = row_bytes / 16;  // 16-byte chunks per row
  const int64_t pieces = (int64_t)n_new * kv.h_kv * 2 * cpr;
  for (int64_t e = tid; e < pieces; e += kAppendThreads) {
    const int c = (int)(e % cpr);
    int64_t r = e / cpr;
    const int which = (int)(r & 1);
    r >>= 1;
    const int g = (int)(r % kv.h_kv);
    const int j = (int)(r / kv.h_kv);
    const int t = L + j;
    const int32_t p = __ldg(kv.page_table + (int64_t)b * kv.max_pages + (t >> kv.log2_ps));
    const int64_t dst = ((((int64_t)p * 2 + which) * kv.h_kv + g) * kv.page_size + (t & (kv.page_size - 1))) * row_bytes;
    const int64_t src = ((((int64_t)b * n_new + j) * kv.h_kv) + g) * row_bytes;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>((which ? v_new : k_new) + src) + c);
    reinterpret_cast<uint4 *>(pool + dst)[c] = v;
  }
}

// seq_lens[b] += delta[b] when the result stays in [0, max_seq_len]; otherwise unchanged and flagged.
__global__ void kv_advance_kernel(int32_t *seq_lens, const int32_t *delta, int batch, int max_seq_len,
                                  unsigned *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  pdl_wait();
  if (b >= batch) return;
  const int64_t v = (int64_t)seq_lens[b] + delta[b];
  if (v >= 0 && v <= max_seq_len)
    seq_lens[b] = (int32_t)v;
  else
    atomicOr(status, (unsigned)SSD_FAULT_SEQLEN);
}

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_kv_append(const ssd_paged_kv *kv, const void *k_new, const void *v_new, int n_new,
                             ssd_stream_t stream) {
  const char *who = "ssd_kv_append";
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if (n_new < 0) return fail(SSD_ERR_INVALID_ARG, "%s: n_new %d < 0", who, n_new);
  if (kv->batch == 0 || n_new == 0) return SSD_OK;
  if (!k_new || !v_new) return fail(SSD_ERR_INVALID_ARG, "%s: k_new and v_new must be non-NULL", who);
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(SSD_ERR_INVALID_ARG, "%s: k_new and v_new must be 16-byte aligned", who);
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  const int row_bytes = kv->d * (kv->dtype == SSD_DTYPE_BF16 ? 2 : 4);
  return launch(kv_append_kernel, dim3(kv->batch), dim3(kAppendThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                "kv_append_kernel", v, static_cast<char *>(const_cast<void *>(kv->pool)),
                static_cast<const char *>(k_new), static_cast<const char *>(v_new), n_new, row_bytes, status);
}

extern "C" int ssd_kv_advance(int32_t *seq_lens, const int32_t *delta, int batch, int max_seq_len,
                              ssd_stream_t stream) {
  const char *who = "ssd_kv_advance";
  if (batch < 0 || max_seq_len < 0) return fail(SSD_ERR_INVALID_ARG, "%s: batch and max_seq_len must be >= 0", who);
  if (batch == 0) return SSD_OK;
  if (!seq_lens || !delta) return fail(SSD_ERR_INVALID_ARG, "%s: seq_lens and delta must be non-NULL", who);
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  return launch(kv_advance_kernel, dim3(cdiv(batch, 256)), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                "kv_advance_kernel", seq_lens, delta, batch, max_seq_len, status);
}
