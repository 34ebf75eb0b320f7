// ssd_unified.cu -- one call that runs verify work for the verify-phase requests and draft work
// for the draft-phase requests of a mixed batch.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.2: the unified batch scheduler mixes requests of both phases in every step
// (about 1/(k+1) of them verify), and a persistent-style fused attention kernel dispatches verify
// and draft attention to their own tile code on chip instead of launching two kernels.
//
// Where the tcgen05 verify applies (bf16, d = 128, pages of 8 or more tokens), the call launches the
// verify over the verify-phase requests (its blocks skip draft-phase requests), the draft kernel
// over the draft-phase requests (its blocks skip verify-phase requests) and then the finalize.  The
// tcgen05 verify holds all of an SM's shared memory, so verify and draft work cannot share a block;
// instead the draft kernel does not wait for the verify (programmatic dependent launch): its blocks
// start once the verify has handed out its last item and run on the SMs the verify's finishing
// blocks leave, so the draft work fills the verify's tail (one mma.sync launch mixing both measured
// about twice the time of separate launches).
// Otherwise one persistent launch mixes both: each block enumerates the work of the whole batch
// itself (per-request item counts and prefix sums in shared memory: verify items first, draft items
// after them, so the long items are started first) and then takes items c, c + grid, c + 2*grid, ...;
// verify items run the mma.sync split tile, draft items the gather tile.  In both forms the
// verify-phase requests then go through the same finalize pass as ssd_verify_attn.
#include "ssd_draft_tile.cuh"
#include "ssd_host.h"
#include "ssd_verify_tile.cuh"

namespace ssd {

int draft_gmax(int G);
size_t draft_data_bytes(int units, int C_max, int gmax, int D);
void draft_carve(unsigned *counters, void *data, int units, int C_max, int gmax, int D, DraftArgs &a);
int draft_checks(const ssd_paged_kv *kv, int h_q, const void *q, const int32_t *idx, int k_max, const int32_t *cnt,
                 const float *out, const char *who, bool need_idx = true);
int launch_draft_any(int dtype, int D, const DraftArgs &a, dim3 grid, cudaStream_t st);
bool verify_tc_supported(const ssd_paged_kv *kv, int R);
int launch_verify_tc(const ssd_paged_kv *kv, const VerifyArgs &a, cudaStream_t st, int max_blocks = 0);

constexpr int kUniMaxBatch = 512;

// SMs left to the draft work while the tensor-core verify runs (ssd_unified_attn): the draft's share
// of the SM time, estimated from the shape alone (the phases and lists are on the device).  A round
// has n_cand - 1 draft phases per verify phase, each reading about k_max / max_seq_len of what a
// verify reads; the draft's SM time is taken as r = 0.9 (n_cand - 1) k_max / max_seq_len of the
// verify's, the factor fitted on the Qwen3-14B mixed batch (64 requests, k = 4, lists of 5 %): 16,
// 24, 33, 40 and 56 draft SMs gave 279.9, 278.6, 283.0, 283.3 and 312.2 us per call, none 290.2.
// Both kinds of work are bound by each SM's latency, not by the HBM, so the split moves SM time
// rather than creating it: the gain is the verify's tail and the draft's launch, both filled.
static int unified_draft_sms(const ssd_paged_kv *kv, int n_cand, int k_max) {
  if (kv->max_seq_len <= 0) return 0;
  const double r = 0.9 * (n_cand - 1) * (double)k_max / kv->max_seq_len;
  const int sm = sm_count();
  int n = (int)(sm * r / (1.0 + r) + 0.5);
  return n < 0 ? 0 : (n > sm / 2 ? sm / 2 : n);
}

template <int D, int NRT, int GMAX>
struct UniCfg {
  static constexpr int V = VerifyMmaCfg<D, NRT>::SMEM;
  static constexpr int Dr = DraftCfg<D, __nv_bfloat16, GMAX>::SMEM;
  static constexpr int SMEM = V > Dr ? V : Dr;
};

template <int D, int NRT, int GMAX>
__global__ void __launch_bounds__(128, 2) unified_kernel(VerifyArgs va, DraftArgs da, const uint8_t *phase) {
  extern __shared__ __align__(128) char smem[];
  __shared__ int s_vpre[kUniMaxBatch + 1];
  __shared__ int s_dpre[kUniMaxBatch + 1];
  const int B = va.kv.batch, h_kv = va.kv.h_kv, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  // Items per request.
  for (int b = tid; b < B; b += blockDim.x) {
    int L = va.kv.seq_lens[b];
    L = L < 0 ? 0 : (L > va.kv.max_seq_len ? va.kv.max_seq_len : L);
    int nv = 0, nd = 0;
    if (phase[b]) {
      nv = h_kv * verify_splits(L);
    } else {
      for (int g = 0; g < h_kv; ++g) {
        int c = da.cnt[b * h_kv + g];
        c = c < 0 ? 0 : (c > da.k_max ? da.k_max : c);
        nd += draft_chunks(c);
      }
    }
    s_vpre[b + 1] = nv;
    s_dpre[b + 1] = nd;
  }
  __syncthreads();
  if (tid == 0) {
    s_vpre[0] = 0;
    s_dpre[0] = 0;
    for (int b = 0; b < B; ++b) {
      s_vpre[b + 1] += s_vpre[b];
      s_dpre[b + 1] += s_dpre[b];
    }
  }
  __syncthreads();
  const int NV = s_vpre[B], ND = s_dpre[B];
  for (int item = blockIdx.x; item < NV + ND; item += gridDim.x) {
    if (item < NV) {
      int lo = 0, hi = B;  // last b with s_vpre[b] <= item
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s_vpre[mid] <= item) lo = mid; else hi = mid;
      }
      const int b = lo, r = item - s_vpre[b];
      int L = va.kv.seq_lens[b];
      L = L < 0 ? 0 : (L > va.kv.max_seq_len ? va.kv.max_seq_len : L);
      const int ns = verify_splits(L);
      verify_item_mma<D, NRT, false>(va, b * h_kv + r / ns, r % ns, smem);
    } else {
      const int i = item - NV;
      int lo = 0, hi = B;
      while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (s_dpre[mid] <= i) lo = mid; else hi = mid;
      }
      const int b = lo;
      int r = i - s_dpre[b], g = 0;
      for (; g < h_kv; ++g) {
        int c = da.cnt[b * h_kv + g];
        c = c < 0 ? 0 : (c > da.k_max ? da.k_max : c);
        int nc = draft_chunks(c);
        if (r < nc) break;
        r -= nc;
      }
      draft_item<D, __nv_bfloat16, GMAX>(da, b * h_kv + g, r, smem);
    }
    __syncthreads();  // the next item reuses shared memory
  }
}

struct UniLayout {
  size_t v_o, v_lse, v_sp, v_sm, split_off, d_off, total;
  int G, R, units, S_max, Lpad, C_max, gmax;
};

static UniLayout uni_layout(const ssd_paged_kv *kv, int h_q, int n_cand, int k_max) {
  UniLayout l{};
  l.G = h_q / kv->h_kv;
  l.R = l.G * n_cand;
  l.units = kv->batch * kv->h_kv;
  l.S_max = cdiv(kv->max_seq_len, kSplitTokens);
  l.Lpad = cdiv(kv->max_seq_len > 0 ? kv->max_seq_len : 1, kSideAlign) * kSideAlign;
  l.C_max = cdiv(k_max > 0 ? k_max : 1, kDraftChunk);
  l.gmax = draft_gmax(l.G);
  Carver c(nullptr);
  c.take<unsigned>(kCounterSlots);  // counter area: verify item counters (slots 0-1), draft arrivals (2 ..)
  size_t rows = (size_t)l.units * l.S_max * l.R;
  l.v_o = c.off;
  c.take<float>(rows * kv->d);
  l.v_lse = c.off;
  c.take<float>(rows);
  l.v_sp = c.off;
  c.take<__half>((size_t)l.units * l.R * l.Lpad);
  l.v_sm = c.off;
  c.take<float>((size_t)l.units * l.R * (l.Lpad / kRefGroup));
  l.split_off = c.off;
  c.take<int>(2);  // split length, first request of the half-length tail
  l.d_off = c.off;
  l.total = l.d_off + draft_data_bytes(l.units, l.C_max, l.gmax, kv->d);
  return l;
}

template <int D, int NRT, int GMAX>
static int launch_uni(const VerifyArgs &va, const DraftArgs &da, const uint8_t *phase, cudaStream_t st) {
  constexpr int smem = UniCfg<D, NRT, GMAX>::SMEM;
  int rc = ensure_smem<unified_kernel<D, NRT, GMAX>>(smem);
  if (rc) return rc;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, unified_kernel<D, NRT, GMAX>, 128, smem);
  const int grid = sm_count() * (per_sm > 0 ? per_sm : 1);
  return launch(unified_kernel<D, NRT, GMAX>, dim3(grid), dim3(128), smem, st, "unified_kernel", va, da, phase);
}

template <int D, int NRT>
static int uni_g(int gmax, const VerifyArgs &va, const DraftArgs &da, const uint8_t *phase, cudaStream_t st) {
  if (gmax == 4) return launch_uni<D, NRT, 4>(va, da, phase, st);
  if (gmax == 8) return launch_uni<D, NRT, 8>(va, da, phase, st);
  return launch_uni<D, NRT, 16>(va, da, phase, st);
}

template <int D>
static int uni_rows(int nrt, int gmax, const VerifyArgs &va, const DraftArgs &da, const uint8_t *phase, cudaStream_t st) {
  if (nrt == 1) return uni_g<D, 1>(gmax, va, da, phase, st);
  if (nrt == 2) return uni_g<D, 2>(gmax, va, da, phase, st);
  return uni_g<D, 4>(gmax, va, da, phase, st);
}

}  // namespace ssd

using namespace ssd;

extern "C" size_t ssd_unified_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand, int k_max) {
  if (!kv || kv->h_kv <= 0 || h_q <= 0 || n_cand <= 0 || k_max < 0 || kv->batch < 0 || kv->max_seq_len < 0 ||
      (kv->d != 64 && kv->d != 128))
    return 0;
  return uni_layout(kv, h_q, n_cand, k_max).total;
}

extern "C" int ssd_unified_attn(const ssd_paged_kv *kv, const uint8_t *phase, const void *q_verify, const void *q_draft,
                                int h_q, int n_cand, const int32_t *idx, int k_max, const int32_t *cnt, float scale,
                                float *out_verify, float *lse_verify, float *scores, int64_t scores_stride,
                                float *out_draft, float *lse_draft, void *workspace, size_t workspace_bytes,
                                ssd_stream_t stream) {
  const char *who = "ssd_unified_attn";
  KVView v;
  int rc = validate_kv(kv, &v, who);
  if (rc) return rc;
  if (!phase) return fail(SSD_ERR_INVALID_ARG, "%s: phase is NULL", who);
  if (kv->dtype != SSD_DTYPE_BF16) return fail(SSD_ERR_UNSUPPORTED, "%s: bf16 caches only", who);
  if ((rc = draft_checks(kv, h_q, q_draft, idx, k_max, cnt, out_draft, who))) return rc;
  if (!q_verify || !out_verify) return fail(SSD_ERR_INVALID_ARG, "%s: q_verify and out_verify must be non-NULL", who);
  if (n_cand < 1) return fail(SSD_ERR_INVALID_ARG, "%s: n_cand < 1", who);
  if ((h_q / kv->h_kv) * n_cand > kMaxRows) return fail(SSD_ERR_UNSUPPORTED, "%s: G*n_cand > %d", who, kMaxRows);
  if (!aligned16(q_verify)) return fail(SSD_ERR_INVALID_ARG, "%s: q_verify must be 16-byte aligned", who);
  if (kv->batch > kUniMaxBatch) return fail(SSD_ERR_UNSUPPORTED, "%s: batch %d > %d", who, kv->batch, kUniMaxBatch);
  if (scores && scores_stride < kv->max_seq_len) return fail(SSD_ERR_INVALID_ARG, "%s: scores_stride too small", who);
  const UniLayout lay = uni_layout(kv, h_q, n_cand, k_max);
  if (!workspace || workspace_bytes < lay.total)
    return fail(SSD_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", who, workspace_bytes, lay.total);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  if (kv->batch == 0 || kv->max_seq_len == 0) return SSD_OK;
  unsigned *status = device_status();
  if (!status) return SSD_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);

  VerifyArgs va{};
  va.kv = v;
  va.q = q_verify;
  va.h_q = h_q;
  va.n_c = n_cand;
  va.G = lay.G;
  va.R = lay.R;
  va.scale_log2 = scale * kLog2e;
  va.S_max = lay.S_max;
  va.Lpad = lay.Lpad;
  va.o_parts = reinterpret_cast<float *>(ws + lay.v_o);
  va.lse_parts = reinterpret_cast<float *>(ws + lay.v_lse);
  va.side_p = scores ? reinterpret_cast<__half *>(ws + lay.v_sp) : nullptr;
  va.side_m = scores ? reinterpret_cast<float *>(ws + lay.v_sm) : nullptr;
  va.status = status;
  DraftArgs da{};
  da.kv = v;
  da.q = q_draft;
  da.h_q = h_q;
  da.G = lay.G;
  da.k_max = k_max;
  da.idx = idx;
  da.cnt = cnt;
  da.scale_log2 = scale * kLog2e;
  da.C_max = lay.C_max;
  da.out = out_draft;
  da.lse = lse_draft;
  da.phase = phase;
  da.status = status;
  const bool tc = verify_tc_supported(kv, lay.R);
  // The draft counters start at slot 2 of the counter area in the three-launch form (slots 0-1 are
  // the tcgen05 verify's item counters).
  draft_carve(reinterpret_cast<unsigned *>(ws) + (tc ? 2 : 0), ws + lay.d_off, lay.units, lay.C_max, lay.gmax, kv->d,
              da);
  if (tc) {
    va.phase = phase;
    va.sched = reinterpret_cast<int *>(ws);
    va.split_out = reinterpret_cast<int *>(ws + lay.split_off);
    // The draft work needs nothing the verify writes, so the two run side by side: the verify takes
    // all SMs but unified_draft_sms() of them and lets the next kernel launch at once; the draft
    // kernel, launched right behind it without waiting for it, runs on the SMs left free and on those
    // the verify's finishing blocks leave.  The finalize follows once both are done.
    const int dsm = pdl_enabled() ? unified_draft_sms(kv, n_cand, k_max) : 0;
    va.early_trigger = dsm > 0;
    if ((rc = launch_verify_tc(kv, va, st, sm_count() - dsm))) return rc;
    da.defer_wait = 1;
    if ((rc = launch_draft_any(kv->dtype, kv->d, da, dim3(lay.C_max, lay.units), st))) return rc;
  } else {
    const int nrt = lay.R <= 16 ? 1 : (lay.R <= 32 ? 2 : 4);
    rc = kv->d == 128 ? uni_rows<128>(nrt, lay.gmax, va, da, phase, st) : uni_rows<64>(nrt, lay.gmax, va, da, phase, st);
    if (rc) return rc;
  }

  FinalizeArgs f{};
  f.seq_lens = kv->seq_lens;
  f.max_seq_len = kv->max_seq_len;
  f.h_kv = kv->h_kv;
  f.h_q = h_q;
  f.n_c = n_cand;
  f.G = lay.G;
  f.R = lay.R;
  f.D = kv->d;
  f.S_max = lay.S_max;
  f.Lpad = lay.Lpad;
  f.o_parts = va.o_parts;
  f.lse_parts = va.lse_parts;
  f.side_p = va.side_p;
  f.side_m = va.side_m;
  f.phase = phase;
  f.out = out_verify;
  f.lse = lse_verify;
  f.scores = scores;
  f.scores_stride = scores_stride;
  f.split_len = tc ? va.split_out : nullptr;
  f.balanced = tc ? 1 : 0;
  f.ref_shift = tc ? kTcRefShift : kRefShift;
  const int n_tok = scores ? cdiv(kv->max_seq_len, kFinTok) : 0;
  return launch_finalize(f, n_tok, lay.units, st);
}
