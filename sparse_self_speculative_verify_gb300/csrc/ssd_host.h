// ssd_host.h -- host-side helpers shared by the libssd translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stddef.h>
#include <stdint.h>

#include "ssd.h"
#include "ssd_common.cuh"

namespace ssd {

// Records a formatted message as the calling thread's last error and returns `code`.
int fail(int code, const char *fmt, ...);
// Maps a pending CUDA launch error to SSD_ERR_CUDA (clearing it); SSD_OK otherwise.
int check_launch(const char *what);
// Device status word of the current device (nullptr + error message on failure).
unsigned *device_status();
// Number of SMs of the current device (cached).
int sm_count();
// Validates the cache description; fills `v`.  `need_mask` lists the accepted dtypes as bits.
int validate_kv(const ssd_paged_kv *kv, KVView *v, const char *who);

// Whether kernels are launched with programmatic stream serialization (programmatic dependent
// launch): on unless the environment variable SSD_PDL is "0" when the library first launches.
bool pdl_enabled();

// Launches kernel<<<grid, block, smem, st>>>(args...) through cudaLaunchKernelEx, with the
// programmatic-stream-serialization attribute when pdl_enabled() (every kernel of the library calls
// pdl_wait() before touching data an earlier kernel may write).  Maps a launch failure to
// SSD_ERR_CUDA with `name` in the message.
template <typename... KArgs, typename... Args>
int launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const char *name,
           Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SSD_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  }
  return check_launch(name);
}

// Raises the dynamic shared-memory limit of `Kernel` to at least `bytes` on the current device;
// the attribute call is made only when the limit has to grow, so launches during CUDA-graph
// capture (after an eager warm-up) make no attribute calls.
template <auto Kernel>
int ensure_smem(int bytes) {
  static int set_bytes[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return fail(SSD_ERR_CUDA, "no current CUDA device");
  }
  if (set_bytes[dev] >= bytes) return SSD_OK;
  cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(SSD_ERR_CUDA, "cudaFuncSetAttribute(%d bytes): %s", bytes, cudaGetErrorString(e));
  }
  set_bytes[dev] = bytes;
  return SSD_OK;
}

// Every workspace begins with a counter area: kCounterSlots 32-bit counters for arrival counting
// and work distribution, at offsets that depend on nothing but the counter's index.  Nothing else is
// stored there and every kernel returns the counters it used to zero when it completes, so a
// workspace zero-filled once stays valid for any later sequence of calls, of any entry point and
// shape.  (Data regions move with the shape; counters placed among them would not stay zero.)
constexpr int kCounterSlots = 65536;
constexpr size_t kCounterBytes = size_t(kCounterSlots) * 4;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Carves consecutive 256-byte aligned regions out of a workspace.
struct Carver {
  char *base;
  size_t off = 0;
  explicit Carver(void *p) : base(static_cast<char *>(p)) {}
  template <typename T>
  T *take(size_t count) {
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off = align256(off + count * sizeof(T));
    return p;
  }
};

}  // namespace ssd
