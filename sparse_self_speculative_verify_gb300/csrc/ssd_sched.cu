// ssd_sched.cu -- phase assignment for the unified verify/draft batch.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.2, workload-aware scheduling: requests of both phases are mixed evenly in
// every step; a greedy bin-packing keeps one bucket per phase and puts each arriving request in the
// least loaded one.  Here a bucket is a phase offset o in [0, k]: at step s the request is in phase
// (s + o) mod (k + 1), the last phase being its verify and the others its k drafts, so balanced
// buckets give every step about B / (k + 1) verifying requests.  Ties go to the lowest offset.
#include "ssd_host.h"

namespace ssd {

__global__ void phase_fill_kernel(const int32_t *offsets, int batch, int n_buckets, int64_t step, uint8_t *phase,
                                  unsigned *status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_trigger();
  pdl_wait();
  if (b >= batch) return;
  const int o = offsets[b];
  if (o < 0 || o >= n_buckets) {  // not a valid offset: treat the request as drafting, flag it
    atomicOr(status, (unsigned)SSD_FAULT_INDEX);
    phase[b] = 0;
    return;
  }
  phase[b] = (uint8_t)(((step + o) % n_buckets) == n_buckets - 1);
}

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_phase_assign(int32_t *counts, int n_buckets, int n_new, int32_t *offset_out) {
  const char *who = "ssd_phase_assign";
  if (!counts || n_buckets <= 0) return fail(SSD_ERR_INVALID_ARG, "%s: counts must be non-NULL, n_buckets > 0", who);
  if (n_new < 0 || (n_new > 0 && !offset_out)) return fail(SSD_ERR_INVALID_ARG, "%s: bad n_new / offset_out", who);
  for (int r = 0; r < n_new; ++r) {
    int best = 0;
    for (int o = 1; o < n_buckets; ++o)
      if (counts[o] < counts[best]) best = o;
    counts[best] += 1;
    offset_out[r] = best;
  }
  return SSD_OK;
}

extern "C" int ssd_phase_fill(const int32_t *offsets, int batch, int n_buckets, int64_t step, uint8_t *phase,
                              ssd_stream_t stream) {
  const char *who = "ssd_phase_fill";
  if (batch < 0 || n_buckets <= 0 || step < 0)
    return fail(SSD_ERR_INVALID_ARG, "%s: batch >= 0, n_buckets > 0 and step >= 0 required", who);
  if (batch == 0) return SSD_OK;
  if (!offsets || !phase) return fail(SSD_ERR_INVALID_ARG, "%s: offsets and phase must be non-NULL", who);
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  return launch(phase_fill_kernel, dim3(cdiv(batch, 256)), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                "phase_fill_kernel", offsets, batch, n_buckets, step, phase, status);
}
