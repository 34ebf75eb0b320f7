// ssd_draft.cu -- sparse draft attention (SparseSpec §4.1: the k drafts after a verify attend only
// the tokens it selected; §4.2: sparse attention = PagedAttention over a token list).
#include "ssd_draft_tile.cuh"
#include "ssd_host.h"

namespace ssd {

// One block per (chunk, unit).  With defer_wait (the unified call, launched right behind the verify
// kernel it does not depend on): no block waits for the previous grid before its work, so the
// draft blocks run on the SMs the verify's finishing blocks leave; block (0, 0) alone waits for it
// before exiting, so that this grid still completes after the verify, and the finalize launched
// behind it (which waits for this grid) sees the verify's results.
template <int D, typename T, int GMAX>
__global__ void __launch_bounds__(128) draft_kernel(DraftArgs a) {
  extern __shared__ __align__(128) char smem[];
  const bool waiter = a.defer_wait && blockIdx.x == 0 && blockIdx.y == 0;
  if (!a.defer_wait) pdl_wait();
  if (!(a.phase && a.phase[blockIdx.y / a.kv.h_kv] != 0))  // not a verify-phase request of a mixed batch
    draft_item<D, T, GMAX>(a, blockIdx.y, blockIdx.x, smem);
  if (waiter) pdl_wait();
}

int draft_gmax(int G) { return G <= 4 ? 4 : (G <= 8 ? 8 : 16); }

// Reading the row pack of a bf16 cache: one block per (request, KV head).
template <int D, int GMAX>
__global__ void __launch_bounds__(128) draft_pack_kernel(DraftArgs a) {
  extern __shared__ __align__(128) char smem[];
  draft_pack_unit<D, GMAX>(a, blockIdx.x, smem);
}

template <int D, int GMAX>
static int launch_draft_pack(const DraftArgs &a, int units, cudaStream_t st) {
  constexpr int smem = DraftPackCfg<D, GMAX>::SMEM;
  int rc = ensure_smem<draft_pack_kernel<D, GMAX>>(smem);
  if (rc) return rc;
  return launch(draft_pack_kernel<D, GMAX>, dim3(units), dim3(128), smem, st, "draft_pack_kernel", a);
}

static int launch_draft_pack_any(int D, const DraftArgs &a, int units, cudaStream_t st) {
  if (!a.pack) return fail(SSD_ERR_INVALID_ARG, "draft: reading the row pack without a pack");
  const int gmax = draft_gmax(a.G);
  if (D == 128)
    return gmax == 4 ? launch_draft_pack<128, 4>(a, units, st)
                     : (gmax == 8 ? launch_draft_pack<128, 8>(a, units, st) : launch_draft_pack<128, 16>(a, units, st));
  return gmax == 4 ? launch_draft_pack<64, 4>(a, units, st)
                   : (gmax == 8 ? launch_draft_pack<64, 8>(a, units, st) : launch_draft_pack<64, 16>(a, units, st));
}

template <int D, typename T, int GMAX>
static int launch_draft(const DraftArgs &a, dim3 grid, cudaStream_t st) {
  constexpr int smem = DraftCfg<D, T, GMAX>::SMEM;
  static_assert(DraftCfg<D, T, GMAX>::TC || 2 * DraftCfg<D, T, GMAX>::TILE >= (128 / (D / 2)) * GMAX * D * 4,
                "reduction area");
  int rc = ensure_smem<draft_kernel<D, T, GMAX>>(smem);
  if (rc) return rc;
  return launch(draft_kernel<D, T, GMAX>, grid, dim3(128), smem, st, "draft_kernel", a);
}

template <int D, typename T>
static int dispatch_g(int gmax, const DraftArgs &a, dim3 grid, cudaStream_t st) {
  if (gmax == 4) return launch_draft<D, T, 4>(a, grid, st);
  if (gmax == 8) return launch_draft<D, T, 8>(a, grid, st);
  return launch_draft<D, T, 16>(a, grid, st);
}

int launch_draft_any(int dtype, int D, const DraftArgs &a, dim3 grid, cudaStream_t st) {
  const int gmax = draft_gmax(a.G);
  if (dtype == SSD_DTYPE_BF16)
    return D == 128 ? dispatch_g<128, __nv_bfloat16>(gmax, a, grid, st) : dispatch_g<64, __nv_bfloat16>(gmax, a, grid, st);
  return D == 128 ? dispatch_g<128, float>(gmax, a, grid, st) : dispatch_g<64, float>(gmax, a, grid, st);
}

// Draft partials: o [units][C_max][GMAX][D], lse [units][C_max][GMAX].  The per-unit arrival
// counters live in the workspace's counter area (slot = unit).
size_t draft_data_bytes(int units, int C_max, int gmax, int D) {
  Carver c(nullptr);
  c.take<float>((size_t)units * C_max * gmax * D);
  c.take<float>((size_t)units * C_max * gmax);
  return c.off;
}

void draft_carve(unsigned *counters, void *data, int units, int C_max, int gmax, int D, DraftArgs &a) {
  Carver c(data);
  a.o_parts = c.take<float>((size_t)units * C_max * gmax * D);
  a.lse_parts = c.take<float>((size_t)units * C_max * gmax);
  a.counters = counters;
}

int draft_checks(const ssd_paged_kv *kv, int h_q, const void *q, const int32_t *idx, int k_max, const int32_t *cnt,
                 const float *out, const char *who, bool need_idx) {
  if (!q || (need_idx && !idx) || !cnt || !out)
    return fail(SSD_ERR_INVALID_ARG, "%s: q, idx, cnt and out must be non-NULL", who);
  if (h_q <= 0 || h_q % kv->h_kv) return fail(SSD_ERR_INVALID_ARG, "%s: h_q %d not a multiple of h_kv", who, h_q);
  if (h_q / kv->h_kv > 16) return fail(SSD_ERR_UNSUPPORTED, "%s: group size %d > 16", who, h_q / kv->h_kv);
  if (k_max < 0) return fail(SSD_ERR_INVALID_ARG, "%s: k_max < 0", who);
  if ((int64_t)kv->batch * kv->h_kv > 65535) return fail(SSD_ERR_UNSUPPORTED, "%s: batch*h_kv above 65535", who);
  return SSD_OK;
}

}  // namespace ssd

using namespace ssd;

extern "C" size_t ssd_draft_workspace_bytes(const ssd_paged_kv *kv, int h_q, int k_max) {
  if (!kv || kv->h_kv <= 0 || h_q <= 0 || k_max < 0 || kv->batch < 0 || (kv->d != 64 && kv->d != 128)) return 0;
  return kCounterBytes + draft_data_bytes(kv->batch * kv->h_kv, cdiv(k_max > 0 ? k_max : 1, kDraftChunk),
                                          draft_gmax(h_q / kv->h_kv), kv->d);
}

// Bytes of the row pack: a K and a V tile of kDraftChunk rows per chunk slot of every unit.
static size_t pack_bytes_of(const ssd_paged_kv *kv, int k_max) {
  const size_t elem = kv->dtype == SSD_DTYPE_BF16 ? 2 : 4;
  return (size_t)kv->batch * kv->h_kv * cdiv(k_max > 0 ? k_max : 1, kDraftChunk) * 2 * kDraftChunk * kv->d * elem;
}

static int draft_call(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max, const int32_t *cnt,
                      float scale, float *out, float *lse, void *pack, size_t pack_bytes, int pack_mode,
                      void *workspace, size_t workspace_bytes, ssd_stream_t stream, const char *who) {
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if (pack_mode != SSD_PACK_NONE && pack_mode != SSD_PACK_WRITE && pack_mode != SSD_PACK_READ &&
      pack_mode != SSD_PACK_READ_DISCARD)
    return fail(SSD_ERR_INVALID_ARG, "%s: pack_mode %d unknown", who, pack_mode);
  const bool discard = pack_mode == SSD_PACK_READ_DISCARD;
  if (discard) pack_mode = SSD_PACK_READ;  // a read, then the pack's lines are dropped
  if ((rc = draft_checks(kv, h_q, q, idx, k_max, cnt, out, who, pack_mode != SSD_PACK_READ))) return rc;
  const size_t need = ssd_draft_workspace_bytes(kv, h_q, k_max);
  if (!workspace || workspace_bytes < need)
    return fail(SSD_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", who, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (pack_mode != SSD_PACK_NONE) {
    const size_t pneed = pack_bytes_of(kv, k_max);
    if (!pack || pack_bytes < pneed)
      return fail(SSD_ERR_WORKSPACE, "%s: row pack %zu bytes, need %zu", who, pack ? pack_bytes : 0, pneed);
    if (reinterpret_cast<uintptr_t>(pack) & 255u)
      return fail(SSD_ERR_INVALID_ARG, "%s: row pack must be 256-byte aligned", who);
  }
  if (kv->batch == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  const int units = kv->batch * kv->h_kv;
  const int C_max = cdiv(k_max > 0 ? k_max : 1, kDraftChunk);
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
  a.pack = pack_mode != SSD_PACK_NONE ? static_cast<char *>(pack) : nullptr;
  a.pack_mode = pack_mode;
  a.pack_discard = discard && kv->dtype == SSD_DTYPE_BF16 ? 1 : 0;  // the fp32 read keeps its lines
  draft_carve(static_cast<unsigned *>(workspace), static_cast<char *>(workspace) + kCounterBytes, units, C_max,
              draft_gmax(a.G), kv->d, a);
  if (pack_mode == SSD_PACK_READ && kv->dtype == SSD_DTYPE_BF16)
    return launch_draft_pack_any(kv->d, a, units, reinterpret_cast<cudaStream_t>(stream));
  return launch_draft_any(kv->dtype, kv->d, a, dim3(C_max, units), reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int ssd_draft_attn(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                              const int32_t *cnt, float scale, float *out, float *lse, void *workspace,
                              size_t workspace_bytes, ssd_stream_t stream) {
  return draft_call(kv, q, h_q, idx, k_max, cnt, scale, out, lse, nullptr, 0, SSD_PACK_NONE, workspace,
                    workspace_bytes, stream, "ssd_draft_attn");
}

extern "C" size_t ssd_draft_pack_bytes(const ssd_paged_kv *kv, int k_max) {
  if (!kv || kv->h_kv <= 0 || k_max < 0 || kv->batch < 0 || (kv->d != 64 && kv->d != 128) ||
      (kv->dtype != SSD_DTYPE_BF16 && kv->dtype != SSD_DTYPE_F32))
    return 0;
  return pack_bytes_of(kv, k_max);
}

extern "C" int ssd_draft_attn_packed(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                                     const int32_t *cnt, float scale, float *out, float *lse, void *pack,
                                     size_t pack_bytes, int pack_mode, void *workspace, size_t workspace_bytes,
                                     ssd_stream_t stream) {
  return draft_call(kv, q, h_q, idx, k_max, cnt, scale, out, lse, pack, pack_bytes, pack_mode, workspace,
                    workspace_bytes, stream, "ssd_draft_attn_packed");
}
