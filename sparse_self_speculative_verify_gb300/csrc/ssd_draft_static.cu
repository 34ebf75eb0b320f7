// ssd_draft_static.cu -- sparse draft attention for callers that cannot hand the library a workspace.
//
// ssd_draft_attn takes its scratch (per-chunk partial outputs, their log-sum-exps and one
// last-arriver counter per (request, KV head)) from a workspace the caller allocates.  Some callers
// have no way to do that at the point where they run the draft step: a plugin inside another
// runtime that owns every device allocation and hands the plugin only its input and output
// buffers, or a serving loop that must not call cudaMalloc / cudaFree while other streams are busy
// (both calls may synchronise the device).  ssd_draft_attn_static runs the same draft kernel with
// its scratch in one fixed-size device array that belongs to this file, so the call needs no
// workspace and allocates nothing.
//
// Costs and rules of that array:
//  * it holds kDraftStaticBytes (16 MiB) on every device that loads the library, until the process
//    exits, whether or not the entry point is ever called;
//  * batches whose scratch would not fit are rejected with SSD_ERR_WORKSPACE before any launch;
//  * every call on a device shares it and it keeps the previous call's contents: the counters that
//    must start at zero are cleared on the call's stream before the kernel runs, and two calls
//    whose work can overlap on the GPU (different streams without ordering between them) race on it;
//  * in host code the array's name is not a device address, so the first call on each device looks
//    the address up with cudaGetSymbolAddress (with that device current) and keeps it; make that
//    first call before any stream capture on the device.
#include <mutex>

#include "ssd_draft_tile.cuh"
#include "ssd_host.h"

namespace ssd {

// Shared with ssd_draft.cu (same kernel, same scratch layout).
int draft_gmax(int G);
size_t draft_data_bytes(int units, int C_max, int gmax, int D);
void draft_carve(unsigned *counters, void *data, int units, int C_max, int gmax, int D, DraftArgs &a);
int draft_checks(const ssd_paged_kv *kv, int h_q, const void *q, const int32_t *idx, int k_max, const int32_t *cnt,
                 const float *out, const char *who, bool need_idx = true);
int launch_draft_any(int dtype, int D, const DraftArgs &a, dim3 grid, cudaStream_t st);

constexpr size_t kDraftStaticBytes = size_t(16) << 20;
static_assert(kDraftStaticBytes == SSD_DRAFT_STATIC_SCRATCH_BYTES, "header and library disagree on the size");

static __device__ __align__(256) unsigned char g_draft_scratch[kDraftStaticBytes];

constexpr int kMaxDevices = 64;
static void *g_scratch_addr[kMaxDevices];  // device address of g_draft_scratch, per device ordinal
static std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once per device.
static int scratch_address(void **out, const char *who) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SSD_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(SSD_ERR_UNSUPPORTED, "%s: device ordinal %d above %d", who, dev, kMaxDevices - 1);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_draft_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return fail(SSD_ERR_CUDA, "%s: cudaGetSymbolAddress of the built-in scratch on device %d: %s", who, dev,
                  cudaGetErrorString(e));
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SSD_OK;
}

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_draft_attn_static(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                                     const int32_t *cnt, float scale, float *out, float *lse, ssd_stream_t stream) {
  const char *who = "ssd_draft_attn_static";
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if ((rc = draft_checks(kv, h_q, q, idx, k_max, cnt, out, who))) return rc;
  const int units = kv->batch * kv->h_kv;
  const int C_max = cdiv(k_max > 0 ? k_max : 1, kDraftChunk);
  const int gmax = draft_gmax(h_q / kv->h_kv);
  // Layout in the array: the per-unit arrival counters, then the partial outputs and their LSEs.
  const size_t ctr_bytes = align256((size_t)units * sizeof(unsigned));
  const size_t need = ctr_bytes + draft_data_bytes(units, C_max, gmax, kv->d);
  if (need > kDraftStaticBytes)
    return fail(SSD_ERR_WORKSPACE,
                "%s: this batch needs %zu bytes of scratch but the built-in scratch holds %zu; use ssd_draft_attn "
                "with a workspace",
                who, need, kDraftStaticBytes);
  if (kv->batch == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  void *scratch = nullptr;
  if ((rc = scratch_address(&scratch, who))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DraftArgs a{};
  a.kv = v;
  a.q = q;
  a.h_q = h_q;
  a.G = h_q / kv->h_kv;
  a.k_max = k_max;
  a.idx = idx;
  a.cnt = cnt;
  a.scale_log2 = scale * kLog2e;
  a.C_max = C_max;
  a.out = out;
  a.lse = lse;
  a.status = status;
  draft_carve(static_cast<unsigned *>(scratch), static_cast<char *>(scratch) + ctr_bytes, units, C_max, gmax, kv->d,
              a);
  // The last-arriver counters must read zero when the kernel starts.
  if (cudaMemsetAsync(a.counters, 0, (size_t)units * sizeof(unsigned), st) != cudaSuccess)
    return check_launch("ssd_draft_attn_static (counter clear)");
  return launch_draft_any(kv->dtype, kv->d, a, dim3(C_max, units), st);
}
