// ssd_host.cu -- error reporting, the device status word and argument validation.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ssd_host.h"

namespace ssd {

static thread_local char t_last_error[512] = "";

// One status word per device; kernels OR fault bits into it (see ssd_device_fault).
__device__ unsigned g_device_status;

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SSD_OK;
}

static constexpr int kMaxDevices = 64;
static unsigned *s_status_ptr[kMaxDevices];
static int s_sm_count[kMaxDevices];

unsigned *device_status() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    fail(SSD_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  if (!s_status_ptr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
    if (e != cudaSuccess) {
      fail(SSD_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
      cudaGetLastError();
      return nullptr;
    }
    s_status_ptr[dev] = static_cast<unsigned *>(p);
  }
  return s_status_ptr[dev];
}

bool pdl_enabled() {
  static const bool on = [] {
    const char *v = getenv("SSD_PDL");
    return !(v && v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 1;
  if (!s_sm_count[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    s_sm_count[dev] = n > 0 ? n : 1;
  }
  return s_sm_count[dev];
}

int validate_kv(const ssd_paged_kv *kv, KVView *v, const char *who) {
  if (!kv) return fail(SSD_ERR_INVALID_ARG, "%s: kv is NULL", who);
  if (!kv->pool || !kv->page_table || !kv->seq_lens)
    return fail(SSD_ERR_INVALID_ARG, "%s: pool, page_table and seq_lens must be non-NULL", who);
  if (kv->dtype != SSD_DTYPE_BF16 && kv->dtype != SSD_DTYPE_F32)
    return fail(SSD_ERR_UNSUPPORTED, "%s: dtype %d (expected SSD_DTYPE_BF16 or SSD_DTYPE_F32)", who, kv->dtype);
  if (kv->d != 64 && kv->d != 128) return fail(SSD_ERR_UNSUPPORTED, "%s: head dim %d (64 or 128)", who, kv->d);
  if (kv->page_size <= 0 || (kv->page_size & (kv->page_size - 1)))
    return fail(SSD_ERR_UNSUPPORTED, "%s: page_size %d is not a power of two", who, kv->page_size);
  if (kv->h_kv <= 0 || kv->batch < 0 || kv->max_pages <= 0 || kv->num_pages <= 0 || kv->max_seq_len < 0)
    return fail(SSD_ERR_INVALID_ARG, "%s: h_kv, max_pages, num_pages must be > 0, batch/max_seq_len >= 0", who);
  if ((int64_t)kv->max_seq_len > (int64_t)kv->max_pages * kv->page_size)
    return fail(SSD_ERR_INVALID_ARG, "%s: max_seq_len %d exceeds max_pages*page_size", who, kv->max_seq_len);
  if (kv->max_seq_len > (1 << 24)) return fail(SSD_ERR_UNSUPPORTED, "%s: max_seq_len above 2^24", who);
  if (!aligned16(kv->pool)) return fail(SSD_ERR_INVALID_ARG, "%s: pool must be 16-byte aligned", who);
  v->pool = kv->pool;
  v->num_pages = kv->num_pages;
  v->page_size = kv->page_size;
  int l2 = 0;
  while ((1 << l2) < kv->page_size) ++l2;
  v->log2_ps = l2;
  v->h_kv = kv->h_kv;
  v->page_table = kv->page_table;
  v->max_pages = kv->max_pages;
  v->seq_lens = kv->seq_lens;
  v->batch = kv->batch;
  v->max_seq_len = kv->max_seq_len;
  return SSD_OK;
}

}  // namespace ssd

extern "C" const char *ssd_last_error(void) { return ssd::t_last_error; }

extern "C" int ssd_version(void) { return (1 << 16) | 0; }

extern "C" int ssd_status(ssd_stream_t stream, uint32_t *status) {
  if (!status) return ssd::fail(SSD_ERR_INVALID_ARG, "ssd_status: status is NULL");
  unsigned *dev = ssd::device_status();
  if (!dev) return SSD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev, sizeof host, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, sizeof(unsigned), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ssd::fail(SSD_ERR_CUDA, "ssd_status: %s", cudaGetErrorString(e));
  }
  *status = host;
  return SSD_OK;
}
