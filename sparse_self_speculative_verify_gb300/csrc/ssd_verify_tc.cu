// ssd_verify_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) verify kernel for bf16 caches with d = 128.
//
// SparseSpec ("Accelerating Large-Scale Reasoning Model Inference: Self-Speculative Decoding with
// Sparse Attention") §4.1: the verify step is full attention of the k+1 candidates over the whole
// cache, and the same kernel dumps what is needed to rematerialise the attention scores (cached
// logits + LSE).  Same work items, partials and criticality side values as the mma.sync tile in
// ssd_verify_tile.cuh; the finalize pass is shared.
//
// One persistent block per SM works through work items (splits of about 512 to 2048 tokens of one
// (request, KV head), whole tiles, equal within a unit: tc_split_count), tile by tile (128 tokens).  Its first item is blockIdx.x; later ones come from a global
// counter, so the items spread over the blocks by how fast each block actually runs.
//  * warp 8 draws the items, hands their numbers to the other warps through a small shared ring, and
//    streams K and V tiles with TMA (one box per page and 64-column panel, 128-byte swizzle, L2
//    evict-first) into a ring of 32 KB slots; the next item's page ids are read one item ahead by
//    the whole warp and each lane issues its own boxes.  Every box goes through TMA: a request's
//    partial last page whole (the softmax masks its K rows past the end and zeroes its V rows),
//    boxes past the end or of skipped pages from a row past the pool, which TMA fills with zeros.
//    The item's query rows arrive by one 4-D TMA box per 64-column panel.
//  * one thread of warp 9 issues   S^T[t][r] = K[t][:] . Q[r][:]      (M = 128 tokens, N = NP)
//    and one thread of warp 10      O^T[d][n] += V[:][d] . P^T[:][n]   (M = 128 = d,   N = 2 NP)
//    where n < NP carries the bf16 high part of the probabilities and n >= NP the bf16 residual, so
//    P keeps about 16 bits.  S is double-buffered in TMEM.  With one issuer per product, QK of a tile
//    goes out as soon as its K tile has landed and its S buffer is free, and PV as soon as its
//    probabilities are in shared memory and its V tile has landed: neither waits behind the other,
//    and V slots return to the producer sooner.
//  * warps 0-3 and 4-7 are two softmax warpgroups: TMEM lane t is token t of the tile (for S) and
//    head dimension d = t (for O); warpgroup w owns rows [w*NP/2, (w+1)*NP/2).  The two groups are
//    independent (rows never mix), so each scheduler runs two softmax warps.
//  * The softmax keeps a lazily updated per-row reference m_ref (log2 domain): probabilities are
//    2^(s - m_ref) <= 2^8; only when a logit exceeds m_ref + 8 does a group agree on a new reference
//    (warp vote, then a transposed warp reduction) and rescale its running sums and its columns of
//    the TMEM accumulator.  Padded rows carry m_ref = +inf, so full tiles need no masking.  The fp16
//    side values for the criticality are these probabilities, stored row-major per (request, KV
//    head) as [row][token], with m_ref stored once per 16 tokens.
//  * All waits are bounded (about one second); on expiry the block raises SSD_FAULT_TIMEOUT in the
//    status word, drains its own copies and MMAs, frees its tensor memory and exits.  Abort
//    decisions are warp-uniform, and the softmax groups synchronise through mbarriers (bounded), not
//    hardware named barriers.
#include "ssd_host.h"
#include "ssd_sm100.cuh"
#include "ssd_verify_tile.cuh"

namespace ssd {
using namespace sm100;

// Timeline record of the diagnostic build (-DSSD_VERIFY_TRACE, trace_verify.py): per block,
// [0] global timer at entry, [1] SM cycles to the end of the prologue, [2] global timer at exit,
// [3] items done, then per item j < kTraceItems: [4 + 3j] cycles when the producer starts the item's
// tiles, [5 + 3j] item number << 32 | tiles, [6 + 3j] cycles when the first softmax warp has
// written its outputs; [127] cycles at exit.  Cycles count from the block's entry.
#ifdef SSD_VERIFY_TRACE
constexpr int kTraceBlocks = 256, kTraceSlots = 128, kTraceItems = 40;
__device__ unsigned long long g_verify_trace[kTraceBlocks * kTraceSlots];
// Per block and tile i < kTraceTiles of its sequence, cycles from the block's entry: [0] the producer
// has a free slot for the tile's K rows, [1] the MMA issuer has issued QK, [2] the first softmax warp
// has S, [3] it has handed P to the MMA issuer, [4] the MMA issuer has seen the K rows land, [5] the
// V rows, [6] it has issued PV, [7] the producer has a free slot for the V rows, [8] the second
// softmax group's first warp has S, [9] it has handed P, [10] the MMA issuer has seen all of P,
// [11] it has seen the S buffer free for the tile's QK.
constexpr int kTraceTiles = 256, kTT = 12;
__device__ unsigned g_verify_tile_trace[kTraceBlocks * kTraceTiles * kTT];
// Per block, its first kTraceMasked masked tiles (the first softmax warp's view), cycles from entry:
// [0] S seen, [1] past the vote barrier, [2] past the reference update, [3] before the P-buffer wait,
// [4] past it, [5] P handed, [6] tile index i | reference updated << 16 | causal << 17, [7] the
// logits masked (before the vote).
constexpr int kTraceMasked = 16;
__device__ unsigned g_verify_masked_trace[kTraceBlocks * kTraceMasked * 8];
// Per block and item j < kTraceItems, the first softmax warp's epilogue, cycles from entry: [0] start
// (last P handed), [1] the item's O complete, [2] past the row-sum barrier, [3] outputs stored.
__device__ unsigned g_verify_epi_trace[kTraceBlocks * kTraceItems * 4];
// Per block and item j < kTraceItems, the producer's item start, cycles from entry: [0] item
// published, [1] item decoded and page ids of the next one requested, [2] query buffer free,
// [3] the item's last tile issued.
__device__ unsigned g_verify_prod_trace[kTraceBlocks * kTraceItems * 4];
// Per block and tile i < kTraceStage, the first softmax warp's stages, cycles from entry: [0] S seen,
// [1] S read and its buffer released, [2] past the vote barrier, [3] past the reference update,
// [4] probabilities and sums done, [5] side values stored, [6] P buffer free, [7] P handed.
constexpr int kTraceStage = 64;
__device__ unsigned g_verify_stage_trace[kTraceBlocks * kTraceStage * 8];
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define SSD_TRACE(stmt) \
  do {                  \
    stmt;               \
  } while (0)
#else
#define SSD_TRACE(stmt) \
  do {                  \
  } while (0)
#endif

// Stage k of the softmax's tile i (trace build only).
#define SSD_STAGE(k) SSD_TRACE(if (tid == 0 && i < kTraceStage) TS[i * 8 + (k)] = (unsigned)(clock64() - clk0))

constexpr int kTcTile = kTcTileTokens;
constexpr int kTcWarps = 11;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcSoftmax = 256;  // two warpgroups
constexpr int kTcProducerWarp = 8;
constexpr int kTcMmaWarp = 9;   // QK issuer; also allocates the tensor memory
constexpr int kTcPvWarp = 10;   // PV issuer
constexpr int kTcMaxBatch = 1024;
constexpr int kTcItemRing = 8;  // item numbers handed from the producer to the other roles
// Split length: each item ends with an epilogue and a pipeline refill that cost a few thousand
// cycles, so items are made as long as load balance allows: about kTcItemsPerBlock items per block
// over the batch's actual tokens, a multiple of the tile, between kSplitTokens and kTcMaxSplit.
constexpr int kTcItemsPerBlock = 4;
constexpr int kTcMaxSplit = kTcMaxSplitTiles * kTcTile;
constexpr int kSlotBytes = kTcTile * 256;  // one K or V tile: 2 panels x 128 rows x 128 B
constexpr int kPanelBytes = kTcTile * 128;  // P tile: one 64-column panel of 128 rows
// K and V tiles: token t's 128-byte row of 64-column panel p sits at (t / 8) * kGroupBytes + p * 1024
// + (t % 8) * 128 (16-byte chunks XOR-swizzled by t % 8), so a page's rows and both panels land in
// one TMA box; the MMA operands step through the 8-row groups with a 2048-byte stride.
constexpr int kGroupBytes = 2048;
constexpr float kLazy = 8.f;

template <int NP>
struct TcCfg {
  static_assert(NP == 32 || NP == 64, "row padding");
  static constexpr int CW = NP / 2;  // columns (rows of the GQA group) per softmax warpgroup
  static constexpr int NSLOT = NP == 32 ? 5 : 3;
  // K tiles and V tiles stream through two rings of their own (slots [0, NK) and [NK, NSLOT)), each
  // consumed in order by one MMA issuer, so a consumer never waits on a slot whose previous fill it
  // has not itself consumed (the phase parity it waits for cannot alias).  A V tile stays until its
  // PV, after the softmax, so the V ring is the deeper one.
  static constexpr int NK = NP == 32 ? 2 : 1;
  static constexpr int NV = NSLOT - NK;
  static constexpr int P_BYTES = kTcTile * (2 * NP) * 2;
  static constexpr int Q_PANEL = NP * 128;
  static constexpr int Q_BYTES = 2 * Q_PANEL;
  static constexpr int TMEM_COLS = 4 * NP;
  static constexpr int OFF_P = NSLOT * kSlotBytes;
  static constexpr int OFF_Q = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_MISC = OFF_Q + 2 * Q_BYTES;
  // misc: 48 mbarriers, flags and the item ring (numbers, then decoded), per-row arrays, reduction
  // scratch, the per-request item prefix, lengths and split shapes
  static constexpr int MISC = 48 * 8 + 128 + kTcItemRing * 32 + NP * 4 * 2 + 2 * 4 * 32 * 4 + (3 * kTcMaxBatch + 1) * 4;
  static constexpr int SMEM = OFF_MISC + MISC + 1024;
};

struct TcItem {
  int b, g, split, L, t0, t1, ntiles, pad;
};

struct TcSmem {
  uint64_t *full, *empty, *s_full, *s_empty, *p_full, *p_empty, *o_full, *o_empty, *q_full, *q_empty, *drain, *grp;
  uint64_t *item_full;  // [kTcItemRing]
  uint32_t *tmem;
  int *abort;
  int *vote;   // [2 groups][4]
  int *items;  // [kTcItemRing] item numbers in processing order; n_items ends the sequence
  TcItem *ring;  // [kTcItemRing] the items decoded (request, head, split, token range, tiles)
  float *mref, *alpha, *red;  // red: [2 groups][4 warps][32]
  int *pre;  // [B+1] item prefix per request
  int *len;  // [B] clamped sequence lengths
  int *nsx;  // [B] splits per unit | tiles per split (before the remainder) << 16
};

__device__ __forceinline__ uint32_t bar_addr(uint64_t *b) { return smem_u32(b); }

// Item -> (request, head, split): items of request b are pre[b] .. pre[b+1]-1, ordered (head, split);
// nsx[b] holds request b's splits per unit (low 16 bits) and tiles per split before the remainder
// (high bits), as tc_split_range cuts them.  Called by a whole warp (warp-uniform item): a 32-ary
// search over pre (one shared load and one ballot per round), then one division.
__device__ __forceinline__ TcItem tc_decode(int item, const int *pre, const int *len, const int *nsx, int B) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = B;  // request b in [lo, hi) with pre[b] <= item < pre[b + 1]
  while (hi - lo > 1) {
    const int step = cdiv(hi - lo, 32);
    const int idx = lo + (lane + 1) * step;
    const bool le = idx < hi && pre[idx] <= item;
    lo += __popc(__ballot_sync(0xffffffffu, le)) * step;
    hi = min(lo + step, hi);
  }
  TcItem it;
  it.b = lo;
  const int r = item - pre[lo];
  const int x = nsx[lo], ns = x & 0xffff, base = x >> 16;
  it.g = r / ns;
  it.split = r - it.g * ns;
  it.L = len[lo];
  const int T = cdiv(it.L, kTcTile), extra = T - base * ns;
  const int first = it.split * base + min(it.split, extra);
  it.t0 = first * kTcTile;
  it.t1 = min((first + base + (it.split < extra ? 1 : 0)) * kTcTile, it.L);
  it.ntiles = cdiv(it.t1 - it.t0, kTcTile);
  return it;
}

// Reduces v[N] (N = 16 or 32) over the 32 lanes of the warp; afterwards lane l holds the result for
// column l % N.
template <int N, bool MAX>
__device__ __forceinline__ float transpose_reduce(float (&v)[N]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int ofs = 16; ofs >= N; ofs >>= 1) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const float o = __shfl_xor_sync(0xffffffffu, v[k], ofs);
      v[k] = MAX ? fmaxf(v[k], o) : v[k] + o;
    }
  }
#pragma unroll
  for (int ofs = N / 2; ofs >= 1; ofs >>= 1) {
    const bool upper = (lane & ofs) != 0;
#pragma unroll
    for (int k = 0; k < ofs; ++k) {
      const float send = upper ? v[k] : v[k + ofs];
      const float keep = upper ? v[k + ofs] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, ofs);
      v[k] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// Transposes an 8 x 8 matrix of 32-bit words held by eight consecutive lanes (lane i = lane % 8 holds
// row i in v[0..7]): afterwards lane i holds column i.  Three butterfly stages swap the off-diagonal
// blocks of 4, 2 and 1 words with the partner lane i ^ s.
__device__ __forceinline__ void transpose8x8(uint32_t (&v)[8], int i) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
    const bool upper = (i & s) != 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p & s) continue;
      const uint32_t send = upper ? v[p] : v[p + s];
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, s);
      if (upper) v[p] = recv; else v[p + s] = recv;
    }
  }
}

// Bounded arrive-and-wait over the 128 threads of one softmax warpgroup.
__device__ __forceinline__ bool group_sync(uint64_t *bar, volatile int *abort, uint32_t &phase) {
  mbar_arrive(bar_addr(bar));
  const bool ok = mbar_wait(bar_addr(bar), phase, abort);
  phase ^= 1u;
  return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded wait: every lane gets the same verdict, so an aborting warp leaves its loops
// together (no lane is stranded at a warp-collective instruction).
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, volatile int *abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v) {
  if constexpr (N == 16) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
  } else {
    static_assert(N == 32, "16 or 32 columns");
    tmem_ld32(taddr, v);
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float *v) {
  if constexpr (N == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
  } else {
    static_assert(N == 32, "16 or 32 columns");
    tmem_st32(taddr, v);
  }
}

template <int NP>
__global__ void __launch_bounds__(kTcThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap qmap,
                     VerifyArgs a, int box_rows) {
  using C = TcCfg<NP>;
  constexpr int CW = C::CW;
  extern __shared__ __align__(1024) char smem_raw[];
  // Rounded up to 1024 bytes by pointer arithmetic on the shared array, so every derived pointer is
  // still known to address shared memory (plain shared loads and stores, not generic ones).
  char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.kv.batch, h_kv = a.kv.h_kv;
#ifdef SSD_VERIFY_TRACE
  unsigned long long *TR = g_verify_trace + (blockIdx.x % kTraceBlocks) * kTraceSlots;
  unsigned *TT = g_verify_tile_trace + (blockIdx.x % kTraceBlocks) * kTraceTiles * kTT;
  unsigned *TM = g_verify_masked_trace + (blockIdx.x % kTraceBlocks) * kTraceMasked * 8;
  unsigned *TE = g_verify_epi_trace + (blockIdx.x % kTraceBlocks) * kTraceItems * 4;
  unsigned *TP = g_verify_prod_trace + (blockIdx.x % kTraceBlocks) * kTraceItems * 4;
  unsigned *TS = g_verify_stage_trace + (blockIdx.x % kTraceBlocks) * kTraceStage * 8;
  int n_masked = 0;
  unsigned tm_s = 0;
  const long long clk0 = clock64();
  if (tid == 0) {
    TR[0] = global_ns();
    TR[3] = 0;
  }
#endif

  TcSmem s;
  {
    char *m = sm + C::OFF_MISC;
    uint64_t *bars = reinterpret_cast<uint64_t *>(m);
    s.full = bars;
    s.empty = bars + 5;
    s.s_full = bars + 10;
    s.s_empty = bars + 12;
    s.p_full = bars + 14;
    s.p_empty = bars + 16;
    s.o_full = bars + 18;
    s.o_empty = bars + 19;
    s.q_full = bars + 20;
    s.q_empty = bars + 22;
    s.drain = bars + 24;
    s.grp = bars + 25;  // [2]
    s.item_full = bars + 32;
    m += 48 * 8;
    s.tmem = reinterpret_cast<uint32_t *>(m);
    s.abort = reinterpret_cast<int *>(s.tmem + 1);
    s.vote = s.abort + 1;  // [8]
    s.items = s.vote + 8;
    m += 128;
    s.ring = reinterpret_cast<TcItem *>(m);
    m += kTcItemRing * sizeof(TcItem);
    s.mref = reinterpret_cast<float *>(m);
    s.alpha = s.mref + NP;
    s.red = s.alpha + NP;  // 16-byte aligned (float4 reads)
    s.pre = reinterpret_cast<int *>(s.red + 2 * 4 * 32);
    s.len = s.pre + kTcMaxBatch + 1;
    s.nsx = s.len + kTcMaxBatch;
  }

  // Set-up that reads nothing an earlier kernel writes runs before the wait for the previous grid:
  // barriers, tensor memory, descriptor prefetch, zeroed query buffers.
  if (a.early_trigger) pdl_trigger();
  if (tid == 0) {
    *s.abort = 0;
    for (int k = 0; k < 8; ++k) s.vote[k] = 0;
    for (int r = 0; r < NP; ++r) s.mref[r] = r < a.R ? -INFINITY : INFINITY;  // first item's references
    for (int k = 0; k < C::NSLOT; ++k) {
      mbar_init(bar_addr(s.full + k), 1);
      mbar_init(bar_addr(s.empty + k), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_addr(s.s_full + k), 1);
      mbar_init(bar_addr(s.s_empty + k), kTcSoftmax);
      mbar_init(bar_addr(s.p_full + k), kTcSoftmax);
      mbar_init(bar_addr(s.p_empty + k), 1);
      mbar_init(bar_addr(s.q_full + k), 1);
      mbar_init(bar_addr(s.q_empty + k), 1);
      mbar_init(bar_addr(s.grp + k), 128);
    }
    mbar_init(bar_addr(s.o_full), 1);
    mbar_init(bar_addr(s.o_empty), kTcSoftmax);
    mbar_init(bar_addr(s.drain), 2);  // one commit by each MMA issuer
    for (int k = 0; k < kTcItemRing; ++k) mbar_init(bar_addr(s.item_full + k), 1);
    mbar_init_fence();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(smem_u32(s.tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kTcProducerWarp && lane == 0) {
    tma_prefetch_desc(&kvmap);
    tma_prefetch_desc(&qmap);
  }
  // Query buffers start zeroed: the TMA writes rows < R only, padded rows must read as zero.
  for (int e = tid; e < 2 * C::Q_BYTES / 16; e += kTcThreads)
    reinterpret_cast<uint4 *>(sm + C::OFF_Q)[e] = make_uint4(0, 0, 0, 0);
  pdl_wait();

  // Per-request lengths, the split length, item counts and their prefix (chunked block scan).
  int split_len, tail_from;  // the batch's split length; requests from tail_from on get half-length splits
  {
    constexpr int CH = cdiv(kTcMaxBatch + 1, kTcThreads);
    int loc[CH];
    long long tok = 0;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int b = tid * CH + k;
      int L = 0;
      if (b < B && a.phase && a.phase[b] == 0) {
        s.len[b] = 0;  // a draft-phase request of a mixed batch: no verify items
      } else if (b < B) {
        L = a.kv.seq_lens[b];
        if (L < a.n_c || L > a.kv.max_seq_len) {
          if (blockIdx.x == 0) atomicOr(a.status, (unsigned)SSD_FAULT_SEQLEN);
          L = L < 0 ? 0 : (L > a.kv.max_seq_len ? a.kv.max_seq_len : L);
        }
        s.len[b] = L;
      }
      loc[k] = L;
      tok += L;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) tok += __shfl_xor_sync(0xffffffffu, tok, o);
    __shared__ long long s_wtok[kTcWarps];
    __shared__ int s_wsum[kTcWarps];
    if (lane == 0) s_wtok[warp] = tok;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    {
      long long total = 0;
      for (int w = 0; w < kTcWarps; ++w) total += s_wtok[w];
      long long per = total * h_kv / ((long long)gridDim.x * kTcItemsPerBlock) / kTcTile * kTcTile;
      split_len = (int)min(max(per, (long long)kSplitTokens), (long long)kTcMaxSplit);
    }
    // Item counts and their prefix, in two passes: the first with the batch's split length for every
    // request finds the tail (the shortest suffix of requests whose items fit in one wave of blocks),
    // the second cuts the tail's requests into half-length splits (tc_tail_split).
    int lens[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) lens[k] = loc[k];
    __shared__ int s_tail;
    tail_from = B;
    for (int pass = 0; pass < 2; ++pass) {
      int sum = 0;
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int b = tid * CH + k, sl = tc_tail_split(split_len, b, tail_from);
        const int ns = tc_split_count(lens[k], sl);
        loc[k] = h_kv * ns;
        sum += loc[k];
        if (pass == 1 && b < B && ns > 0) s.nsx[b] = ns | (cdiv(lens[k], kTcTile) / ns) << 16;
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) s_wsum[warp] = incl;
      __syncthreads();
      int off = 0;
      for (int w = 0; w < warp; ++w) off += s_wsum[w];
      off += incl - sum;
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int b = tid * CH + k;
        if (b <= B) s.pre[b] = off;
        off += loc[k];
      }
      __syncthreads();
      if (pass == 1) break;
      // The first b whose suffix of items is at most one per block (b = B qualifies: exactly one does).
      const int total_items = s.pre[B];
#pragma unroll
      for (int k = 0; k < CH; ++k) {
        const int b = tid * CH + k;
        if (b <= B && total_items - s.pre[b] <= (int)gridDim.x && (b == 0 || total_items - s.pre[b - 1] > (int)gridDim.x))
          s_tail = b;
      }
      __syncthreads();
      tail_from = s_tail;
      __syncthreads();  // every thread has read s.pre before the second pass rewrites it
    }
    if (blockIdx.x == 0 && tid == 0) {
      a.split_out[0] = split_len;
      a.split_out[1] = tail_from;
    }
    __syncthreads();
  }
  const uint32_t tm = *s.tmem;
  const int n_items = s.pre[B];
  SSD_TRACE(if (tid == 0) TR[1] = clock64() - clk0);
  const int G = a.G, R = a.R, n_c = a.n_c;

  if (warp == kTcProducerWarp) {
    // ---------------------------------------------------------------- TMA producer + query rows
    // Control flow stays warp-uniform: lane 0 waits, the verdict is broadcast.
    const uint64_t pol = policy_evict_first();
    const int ps = a.kv.page_size, lps = a.kv.log2_ps;
    // First row past the pool (the tensor map's row count; below 2^31, checked on the host).
    const int oob_row = (int)((int64_t)a.kv.num_pages * 2 * h_kv * ps);
    uint32_t nk = 0, nv = 0;  // K and V tiles issued
    int jl = 0;
    bool ok = true;
    // Page ids of an item's boxes, read by the whole warp one item ahead of use: box j (tokens
    // t0 + j*box_rows) lives in lane j % 32, register j / 32 (boxes hold at least 8 rows).
    constexpr int kPidRegs = kTcMaxSplit / (8 * 32);
    // Page ids of item nx's boxes (none when nx is the end marker).
    auto load_pids = [&](const TcItem &nx, bool have, int32_t(&dst)[kPidRegs]) {
#pragma unroll
      for (int h = 0; h < kPidRegs; ++h) {
        const int t = nx.t0 + (h * 32 + lane) * box_rows;
        dst[h] = have && t < nx.t1 ? __ldg(a.kv.page_table + (int64_t)nx.b * a.kv.max_pages + (t >> lps)) : -1;
      }
    };
    // Work distribution: the block's first item is blockIdx.x, every later one is drawn from a global
    // counter (items gridDim.x, gridDim.x + 1, ...), so blocks that run ahead take more items.  The
    // draw for item j+1 is issued after the loads of item j's fourth tile from the end, and item j+1
    // is decoded (tc_decode: a few hundred cycles) and its page ids requested after the loads of its
    // second tile from the end: none of it sits at an item boundary, where the ring would drain, the
    // atomic has two tiles to return, and a block holds a drawn item only for the last tiles of the
    // current one, so the blocks run out of work close together.  Lane 0 holds the raw draw.
    int cur = blockIdx.x;
    int raw = 0;
    TcItem it_cur{};
    if (cur < n_items) it_cur = tc_decode(cur, s.pre, s.len, s.nsx, B);
    int32_t pid_cur[kPidRegs];
    load_pids(it_cur, cur < n_items, pid_cur);
    const int boxes_per_tile = kTcTile / box_rows;
    for (;; ++jl) {
      // Hand the item to the MMA and softmax roles (n_items ends their loops). The slot
      // written here last held item jl - kTcItemRing, which every role has read by now: this warp
      // has passed the query-buffer wait of item jl - 1, so the QK issuer is done with item jl - 3,
      // the softmax warps (which read the S tile two tiles back) have begun item jl - 5 at least,
      // and the PV issuer (at most two tiles behind the softmax) has begun item jl - 7.
      if (lane == 0) {
        s.items[jl % kTcItemRing] = cur;
        s.ring[jl % kTcItemRing] = it_cur;
        mbar_arrive(bar_addr(s.item_full + jl % kTcItemRing));
      }
      SSD_TRACE(if (lane == 0 && jl < kTraceItems) TP[jl * 4] = (unsigned)(clock64() - clk0));
      if (cur >= n_items || !ok) break;
      const TcItem it = it_cur;
      TcItem it_nx{};
      int32_t pid_nx[kPidRegs];
      int nxt = n_items;
      const int k_draw = max(0, it.ntiles - 4), k_next = min(it.ntiles - 1, max(k_draw + 2, it.ntiles - 2));
      SSD_TRACE(if (lane == 0 && jl < kTraceItems) TP[jl * 4 + 1] = (unsigned)(clock64() - clk0));
      // Query rows of this item: one 4-D TMA box per 64-column panel (d x 1 x G heads x n_c
      // candidates lands as rows r = i*G + h, 128-byte swizzled); rows >= R stay zero.
      const bool qok = lane == 0 ? mbar_wait(bar_addr(s.q_empty + (jl & 1)), ((jl >> 1) & 1) ^ 1, s.abort) : true;
      if (!__shfl_sync(0xffffffffu, qok, 0)) { ok = false; break; }
      SSD_TRACE(if (lane == 0 && jl < kTraceItems) TP[jl * 4 + 2] = (unsigned)(clock64() - clk0));
      if (lane == 0) {
        const uint32_t qf = bar_addr(s.q_full + (jl & 1));
        const uint32_t qb = sbase + C::OFF_Q + (jl & 1) * C::Q_BYTES;
        mbar_arrive_expect_tx(qf, 2u * R * 128u);
        tma_load_4d(qb, &qmap, 0, 0, it.g * G, it.b * n_c, qf);
        tma_load_4d(qb + C::Q_PANEL, &qmap, 0, 1, it.g * G, it.b * n_c, qf);
      }
      __syncwarp();
      SSD_TRACE(if (lane == 0 && jl < kTraceItems) {
        TR[4 + 3 * jl] = clock64() - clk0;
        TR[5 + 3 * jl] = ((unsigned long long)cur << 32) | (unsigned)it.ntiles;
      });
      for (int k = 0; ok && k < it.ntiles; ++k) {
        const int tb = it.t0 + k * kTcTile, tend = min(tb + kTcTile, it.t1);
        // Lane j < boxes_per_tile handles box j of this tile.
        const int jb = k * boxes_per_tile + lane;
        int32_t pid = -1;
#pragma unroll
        for (int h = 0; h < kPidRegs; ++h) {
          const int32_t ph = __shfl_sync(0xffffffffu, pid_cur[h], jb & 31);
          if ((jb >> 5) == h) pid = ph;
        }
        const int t = tb + lane * box_rows;
        const bool in_tile = lane < boxes_per_tile;
        const bool page_ok = pid >= 0 && (int64_t)pid < a.kv.num_pages;
        const int nvalid = in_tile ? max(0, min(box_rows, tend - t)) : 0;  // rows of this box in [tb, tend)
        if (nvalid > 0 && !page_ok) atomicOr(a.status, (unsigned)SSD_FAULT_PAGE);
        // Every box of the tile goes through TMA.  A box with rows of the unit on a good page is
        // loaded whole: in the request's partial last page the rows past its end hold whatever the
        // page holds, which the softmax masks (K) and zeroes before PV reads them (V).  Boxes past
        // the end and boxes of skipped pages start at a row past the pool's last, which TMA fills
        // with zeros (no memory traffic).
        const int row_kv0 = nvalid > 0 && page_ok ? (int)((((int64_t)pid * 2) * h_kv + it.g) * ps + (t & (ps - 1)))
                                                   : -1;
        for (int kv = 0; kv < 2; ++kv) {
          const uint32_t f = kv == 0 ? nk : nv;  // this tile's number in the block's sequence
          const int slot = kv == 0 ? (int)(f % C::NK) : C::NK + (int)(f % C::NV);
          const uint32_t use = kv == 0 ? f / C::NK : f / C::NV;
          const bool eok = lane == 0 ? mbar_wait(bar_addr(s.empty + slot), (use & 1) ^ 1, s.abort) : true;
          if (!__shfl_sync(0xffffffffu, eok, 0)) { ok = false; break; }
          SSD_TRACE(if (lane == 0 && f < kTraceTiles) TT[f * kTT + (kv ? 7 : 0)] = (unsigned)(clock64() - clk0));
          const uint32_t fb = bar_addr(s.full + slot);
          if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(boxes_per_tile * box_rows) * 256u);
          __syncwarp();
          if (in_tile) {
            const int row = row_kv0 >= 0 ? row_kv0 + kv * h_kv * ps : oob_row;
            const uint32_t dst = sbase + slot * kSlotBytes + ((t - tb) >> 3) * kGroupBytes;
            tma_load_4d(dst, &kvmap, 0, 0, 0, row >> 3, fb, pol);  // box_rows rows, both panels
          }
          __syncwarp();
          if (kv == 0) ++nk; else ++nv;
        }
        // Look-ahead (see above): the draw, then the drawn item decoded with its page ids.
        if (k == k_draw && lane == 0) raw = atomicAdd(a.sched, 1);
        if (k == k_next) {
          nxt = min((int)gridDim.x + __shfl_sync(0xffffffffu, raw, 0), n_items);
          if (nxt < n_items) it_nx = tc_decode(nxt, s.pre, s.len, s.nsx, B);
          load_pids(it_nx, nxt < n_items, pid_nx);
        }
      }
      SSD_TRACE(if (lane == 0 && jl < kTraceItems) TP[jl * 4 + 3] = (unsigned)(clock64() - clk0));
      it_cur = it_nx;
#pragma unroll
      for (int h = 0; h < kPidRegs; ++h) pid_cur[h] = pid_nx[h];
      cur = nxt;
    }
    // The block has taken its last item: the next kernel on the stream may begin launching.
    pdl_trigger();
    // Every draw this warp issued has returned (also after an abort) before the block counts itself
    // finished below, so the counter reset cannot overtake a draw.
    const int last_draw = __shfl_sync(0xffffffffu, raw, 0);
    asm volatile("" ::"r"(last_draw));
    if (!ok && lane == 0) {
      // Drain: every fill issued so far must land before the block's shared memory is released.
      volatile int never = 0;
      for (uint32_t f = nk > (uint32_t)C::NK ? nk - C::NK : 0; f < nk; ++f)
        mbar_wait(bar_addr(s.full + f % C::NK), (f / C::NK) & 1, &never);
      for (uint32_t f = nv > (uint32_t)C::NV ? nv - C::NV : 0; f < nv; ++f)
        mbar_wait(bar_addr(s.full + C::NK + f % C::NV), (f / C::NV) & 1, &never);
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ---------------------------------------------------------------- QK issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16_f32(128, NP, 0, 0);
      uint32_t i = 0;
      for (int jl = 0;; ++jl) {
        if (!mbar_wait(bar_addr(s.item_full + jl % kTcItemRing), (jl / kTcItemRing) & 1, s.abort)) break;
        const int item = *reinterpret_cast<volatile int *>(s.items + jl % kTcItemRing);
        if (item >= n_items) break;
        const TcItem it = s.ring[jl % kTcItemRing];
        if (!mbar_wait(bar_addr(s.q_full + (jl & 1)), (jl >> 1) & 1, s.abort)) break;
        const uint64_t qd = smem_desc(sbase + C::OFF_Q + (jl & 1) * C::Q_BYTES, 16, 1024);
        bool ok = true;
        for (int k = 0; k < it.ntiles; ++k, ++i) {
          const int kslot = (int)(i % C::NK);
          if (!mbar_wait(bar_addr(s.full + kslot), (i / C::NK) & 1, s.abort)) { ok = false; break; }
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 4] = (unsigned)(clock64() - clk0));
          if (!mbar_wait(bar_addr(s.s_empty + (i & 1)), ((i >> 1) & 1) ^ 1, s.abort)) { ok = false; break; }
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 11] = (unsigned)(clock64() - clk0));
          tc_fence_after();
          // Descriptors of the K step kk: the start address field (bits 0-13, address >> 4) advanced
          // from the tile's base descriptor (addresses stay below 256 KB: no carry out of the field).
          const uint64_t ka = smem_desc(sbase + kslot * kSlotBytes, 16, kGroupBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tm + (i & 1) * NP, ka + (uint64_t)(((kk >> 2) * 1024 + (kk & 3) * 32) >> 4),
                        qd + (uint64_t)(((kk >> 2) * C::Q_PANEL + (kk & 3) * 32) >> 4), id_qk, kk > 0 ? 1u : 0u);
          mma_commit(bar_addr(s.s_full + (i & 1)));
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 1] = (unsigned)(clock64() - clk0));
          mma_commit(bar_addr(s.empty + kslot));
          if (k == it.ntiles - 1) mma_commit(bar_addr(s.q_empty + (jl & 1)));
        }
        if (!ok) break;
      }
      // Drain every MMA this thread issued before the tensor memory is released.
      mma_commit(bar_addr(s.drain));
      volatile int never = 0;
      mbar_wait(bar_addr(s.drain), 0, &never);
    }
    __syncwarp();
  } else if (warp == kTcPvWarp) {
    // ---------------------------------------------------------------- PV issuer
    if (lane == 0) {
      const uint32_t id_pv = idesc_bf16_f32(128, 2 * NP, 1, 1);
      const uint32_t o_col = tm + 2 * NP;
      uint32_t i = 0;
      for (int jl = 0;; ++jl) {
        if (!mbar_wait(bar_addr(s.item_full + jl % kTcItemRing), (jl / kTcItemRing) & 1, s.abort)) break;
        const int item = *reinterpret_cast<volatile int *>(s.items + jl % kTcItemRing);
        if (item >= n_items) break;
        const TcItem it = s.ring[jl % kTcItemRing];
        bool ok = true;
        for (int k = 0; k < it.ntiles; ++k, ++i) {
          const int vslot = C::NK + (int)(i % C::NV);
          if (!mbar_wait(bar_addr(s.full + vslot), (i / C::NV) & 1, s.abort)) { ok = false; break; }
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 5] = (unsigned)(clock64() - clk0));
          if (!mbar_wait(bar_addr(s.p_full + (i & 1)), (i >> 1) & 1, s.abort)) { ok = false; break; }
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 10] = (unsigned)(clock64() - clk0));
          if (k == 0 && !mbar_wait(bar_addr(s.o_empty), (jl & 1) ^ 1, s.abort)) { ok = false; break; }
          tc_fence_after();
          // V^T as an MN-major operand: 64-element d atoms (panels) 1024 bytes apart, 8-token groups
          // kGroupBytes apart; P^T: 64-column panels kPanelBytes apart, 8-token groups 1024 apart.
          const uint64_t vd = smem_desc(sbase + vslot * kSlotBytes, 1024, kGroupBytes);
          const uint64_t pd = smem_desc(sbase + C::OFF_P + (i & 1) * C::P_BYTES, kPanelBytes, 1024);
#pragma unroll
          for (int st = 0; st < kTcTile / 16; ++st)  // token step st: 16 tokens further
            mma_bf16_ss(o_col, vd + (uint64_t)(st * 2 * kGroupBytes >> 4), pd + (uint64_t)(st * 2048 >> 4), id_pv,
                        (k == 0 && st == 0) ? 0u : 1u);
          SSD_TRACE(if (i < kTraceTiles) TT[i * kTT + 6] = (unsigned)(clock64() - clk0));
          mma_commit(bar_addr(s.empty + vslot));
          mma_commit(bar_addr(s.p_empty + (i & 1)));
          if (k == it.ntiles - 1) mma_commit(bar_addr(s.o_full));
        }
        if (!ok) break;
      }
      mma_commit(bar_addr(s.drain));
      volatile int never = 0;
      mbar_wait(bar_addr(s.drain), 0, &never);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int wg = warp >> 2, tw = tid & 127, wiw = warp & 3;  // group, lane of TMEM, warp in group
    const int c0 = wg * CW;                                      // first row of this group
    uint64_t *grp = s.grp + wg;
    int *vote = s.vote + wg * 4;
    float *red = s.red + wg * 4 * 32;
    const uint32_t lane_base = (uint32_t)(wiw * 32) << 16;
    const int nref = ref_stride(a.Lpad, kTcRefShift);
    const uint64_t side_pol = policy_l2_evict_last();
    uint32_t i = 0, gph = 0;
    int jl = 0;
    // The item sequence comes from the producer's ring.  Each item's per-row references start at
    // -inf (padded rows +inf): in shared memory, the thread that owns a row resets it at the end of
    // the previous item (the same thread reads it first in the next item's reference update, and
    // every other reader comes after a group barrier); the first tile takes the start values from
    // registers.  So no group barrier is needed between items.
    int item = n_items;
    TcItem it{};
    if (!wwait(bar_addr(s.item_full), 0, s.abort)) goto out;
    item = *reinterpret_cast<volatile int *>(s.items);
    if (item < n_items) it = s.ring[0];
    for (;; ++jl) {
      if (item >= n_items) break;
      const int u = it.b * h_kv + it.g;
      const int lim_base = it.L - n_c;  // row r sees t <= lim_base + r / G
      float lsum[CW];
#pragma unroll
      for (int j = 0; j < CW; ++j) lsum[j] = 0.f;
      for (int k = 0; k < it.ntiles; ++k, ++i) {
        const int tb = it.t0 + k * kTcTile, t = tb + tw;
        if (!wwait(bar_addr(s.s_full + (i & 1)), (i >> 1) & 1, s.abort)) goto out;
        SSD_TRACE(if (tid == 0 && i < kTraceTiles) TT[i * kTT + 2] = (unsigned)(clock64() - clk0));
        SSD_STAGE(0);
        SSD_TRACE(if (tid == 128 && i < kTraceTiles) TT[i * kTT + 8] = (unsigned)(clock64() - clk0));
        SSD_TRACE(tm_s = (unsigned)(clock64() - clk0));
        tc_fence_after();
        float x[CW];
        tmem_ld_cols<CW>(tm + lane_base + (i & 1) * NP + c0, x);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar_addr(s.s_empty + (i & 1)));
        SSD_STAGE(1);
        // Rows of skipped pages hold zeros in the K/V slots; rows past the unit's end hold zeros or
        // the rest of its last page, so tokens t >= t1 are masked here and their V rows zeroed below.
        const bool valid = t < it.t1;
        const bool causal = tb + kTcTile - 1 > lim_base;
        const bool masked = causal || !__all_sync(0xffffffffu, valid);
        float mr[CW];
        if (k == 0) {
#pragma unroll
          for (int j = 0; j < CW; ++j) mr[j] = c0 + j < R ? -INFINITY : INFINITY;
        } else {
#pragma unroll
          for (int j = 0; j < CW; j += 4) *reinterpret_cast<float4 *>(mr + j) = *reinterpret_cast<const float4 *>(s.mref + c0 + j);
        }
        // d = scale * s - m_ref (log2 domain); -inf where the row cannot see the token.
        float dl[CW];
        if (masked) {
          // Row r sees token t iff t <= lim_base + floor(r / G), i.e. (t - lim_base) G <= r.
          const int tg = causal ? (t - lim_base) * G : INT_MIN;
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const int r = c0 + j;
            const bool vis = valid && r < R && tg <= r;
            x[j] = vis ? x[j] * a.scale_log2 : -INFINITY;
            dl[j] = vis ? x[j] - mr[j] : -INFINITY;  // never -inf - (-inf)
          }
        } else {
#pragma unroll
          for (int j = 0; j < CW; ++j) dl[j] = fmaf(x[j], a.scale_log2, -mr[j]);  // padded rows: -inf
        }
        bool need = false;
#pragma unroll
        for (int j = 0; j < CW; ++j) need |= dl[j] > kLazy;
        SSD_TRACE(if (masked && tid == 0 && n_masked < kTraceMasked) TM[n_masked * 8 + 7] = (unsigned)(clock64() - clk0));
        if (__any_sync(0xffffffffu, need) && lane == 0) vote[i & 3] = 1;
        if (!group_sync(grp, s.abort, gph)) goto out;
        const bool any = vote[i & 3] != 0;
        if (tw == 0) vote[(i + 2) & 3] = 0;
        SSD_STAGE(2);
#ifdef SSD_VERIFY_TRACE
        const bool trace_m = masked && tid == 0 && n_masked < kTraceMasked;
#endif
        SSD_TRACE(if (trace_m) {
          TM[n_masked * 8 + 0] = tm_s;
          TM[n_masked * 8 + 1] = (unsigned)(clock64() - clk0);
          TM[n_masked * 8 + 6] = (unsigned)i | (any ? 1u << 16 : 0u) | (causal ? 1u << 17 : 0u);
        });
        if (any) {
          // New reference: per-row maximum of the tile (over the group's 128 tokens).
          float v[CW];
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const int r = c0 + j;
            if (!masked) x[j] = r < R ? x[j] * a.scale_log2 : -INFINITY;
            v[j] = x[j];
          }
          const float mx = transpose_reduce<CW, true>(v);
          if (lane < CW) red[wiw * 32 + lane] = mx;
          if (!group_sync(grp, s.abort, gph)) goto out;
          if (tw < CW) {
            const int r = c0 + tw;
            const float m_old = s.mref[r];
            const float mt = fmaxf(fmaxf(red[tw], red[32 + tw]), fmaxf(red[64 + tw], red[96 + tw]));
            if (r < R) {
              const float m_new = fmaxf(m_old, mt);
              s.alpha[r] = (m_old == -INFINITY) ? 0.f : fast_exp2(m_old - m_new);
              s.mref[r] = m_new;
            } else {
              s.alpha[r] = 1.f;
            }
          }
          if (!group_sync(grp, s.abort, gph)) goto out;
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            lsum[j] *= s.alpha[c0 + j];
            mr[j] = s.mref[c0 + j];
            dl[j] = (x[j] == -INFINITY) ? -INFINITY : x[j] - mr[j];
          }
          if (k > 0) {
            // Rescale this group's columns of the accumulator once the previous PV has landed.
            const uint32_t pj = i - 1;
            if (!wwait(bar_addr(s.p_empty + (pj & 1)), (pj >> 1) & 1, s.abort)) goto out;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float o[CW];
              const uint32_t col = tm + lane_base + 2 * NP + h * NP + c0;
              tmem_ld_cols<CW>(col, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < CW; ++j) o[j] *= s.alpha[c0 + j];
              tmem_st_cols<CW>(col, o);
            }
            tmem_st_wait();
            tc_fence_before();
          }
        }
        SSD_TRACE(if (trace_m) TM[n_masked * 8 + 2] = (unsigned)(clock64() - clk0));
        SSD_STAGE(3);
        // Probabilities (<= 2^kLazy; exp2(-inf) = 0), running sums, side values, P tile.
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          x[j] = fast_exp2(dl[j]);
          lsum[j] += x[j];
        }
        SSD_STAGE(4);
        if (a.side_p != nullptr) {
          // fp16 side values, row-major per (unit, row).  The eight lanes that hold eight consecutive
          // tokens transpose their (row pair, token) values, so that lane j stores rows 2j and 2j + 1 of
          // each batch of 16 rows for those eight tokens: two 16-byte stores instead of 16 two-byte ones.
          const int j8 = lane & 7;
          __half *sp = a.side_p + (int64_t)u * R * a.Lpad + (t - j8);
#pragma unroll
          for (int hb = 0; hb < CW / 16; ++hb) {
            uint32_t h[8];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const __half2 v = __floats2half2_rn(x[16 * hb + 2 * p], x[16 * hb + 2 * p + 1]);
              h[p] = *reinterpret_cast<const uint32_t *>(&v);
            }
            transpose8x8(h, j8);
            const int r = c0 + 16 * hb + 2 * j8;
            const uint4 lo = make_uint4(__byte_perm(h[0], h[1], 0x5410), __byte_perm(h[2], h[3], 0x5410),
                                        __byte_perm(h[4], h[5], 0x5410), __byte_perm(h[6], h[7], 0x5410));
            const uint4 hi = make_uint4(__byte_perm(h[0], h[1], 0x7632), __byte_perm(h[2], h[3], 0x7632),
                                        __byte_perm(h[4], h[5], 0x7632), __byte_perm(h[6], h[7], 0x7632));
            // Kept in L2 (the criticality pass reads them next and then drops them from L2 unwritten).
            if (r < R) st_global_policy(sp + (int64_t)r * a.Lpad, lo, side_pol);
            if (r + 1 < R) st_global_policy(sp + (int64_t)(r + 1) * a.Lpad, hi, side_pol);
          }
          // References: one per (row, tile), since every value of the tile was taken against the
          // same reference.
          if (tw < CW && c0 + tw < R) {
            const float m = s.mref[c0 + tw];
            a.side_m[((int64_t)u * R + c0 + tw) * nref + (tb >> kTcRefShift)] = (m == -INFINITY) ? 0.f : m;
          }
        }
        SSD_TRACE(if (trace_m) TM[n_masked * 8 + 3] = (unsigned)(clock64() - clk0));
        SSD_STAGE(5);
        if (!wwait(bar_addr(s.p_empty + (i & 1)), ((i >> 1) & 1) ^ 1, s.abort)) goto out;
        SSD_STAGE(6);
        SSD_TRACE(if (trace_m) TM[n_masked * 8 + 4] = (unsigned)(clock64() - clk0));
        {
          char *prow = sm + C::OFF_P + (i & 1) * C::P_BYTES + tw * 128;
#pragma unroll
          for (int c8 = 0; c8 < CW / 8; ++c8) {
            uint32_t h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split_bf16(x[8 * c8 + 2 * e], x[8 * c8 + 2 * e + 1], h[e], l[e]);
            // Columns n = c0 + 8*c8 .. +7 (high part) and NP + c0 + 8*c8 .. (residual); 64 columns
            // per 128-byte swizzle atom.
            const int nh = c0 + 8 * c8, nl = NP + c0 + 8 * c8;
            *reinterpret_cast<uint4 *>(prow + (nh >> 6) * kPanelBytes + ((((nh & 63) >> 3) ^ (tw & 7)) << 4)) =
                make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(prow + (nl >> 6) * kPanelBytes + ((((nl & 63) >> 3) ^ (tw & 7)) << 4)) =
                make_uint4(l[0], l[1], l[2], l[3]);
          }
        }
        if (wg == 0 && !__all_sync(0xffffffffu, valid)) {
          // The tile ends the unit: the first group zeroes the V rows of tokens past the end once
          // the tile has landed (their probabilities are 0, but a stale row could hold NaN bits).
          const int vslot = C::NK + (int)(i % C::NV);
          if (!wwait(bar_addr(s.full + vslot), (i / C::NV) & 1, s.abort)) goto out;
          if (!valid) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              *reinterpret_cast<uint4 *>(sm + vslot * kSlotBytes + (tw >> 3) * kGroupBytes + (c >> 3) * 1024 +
                                         (tw & 7) * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_addr(s.p_full + (i & 1)));
        SSD_TRACE(if (tid == 0 && i < kTraceTiles) TT[i * kTT + 3] = (unsigned)(clock64() - clk0));
        SSD_STAGE(7);
        SSD_TRACE(if (tid == 128 && i < kTraceTiles) TT[i * kTT + 9] = (unsigned)(clock64() - clk0));
        SSD_TRACE(if (trace_m) TM[(n_masked++) * 8 + 5] = (unsigned)(clock64() - clk0));
      }
      // The next item (published by the producer once this item's tiles were issued), decoded while
      // the last PV of this item completes.
      const uint32_t nj = (uint32_t)jl + 1;
      if (!wwait(bar_addr(s.item_full + nj % kTcItemRing), (nj / kTcItemRing) & 1, s.abort)) goto out;
      const int next_item = *reinterpret_cast<volatile int *>(s.items + nj % kTcItemRing);
      TcItem nx{};
      if (next_item < n_items) nx = s.ring[nj % kTcItemRing];
      // Epilogue: O (high + residual columns) and the row sums -> the split's normalised partial.
      {
        SSD_TRACE(if (tid == 0 && jl < kTraceItems) TE[jl * 4] = (unsigned)(clock64() - clk0));
        if (!wwait(bar_addr(s.o_full), jl & 1, s.abort)) goto out;
        SSD_TRACE(if (tid == 0 && jl < kTraceItems) TE[jl * 4 + 1] = (unsigned)(clock64() - clk0));
        tc_fence_after();
        float o[CW];
        {
          float hi[CW], lo[CW];
          tmem_ld_cols<CW>(tm + lane_base + 2 * NP + c0, hi);
          tmem_ld_cols<CW>(tm + lane_base + 3 * NP + c0, lo);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < CW; ++j) o[j] = hi[j] + lo[j];
        }
        tc_fence_before();
        mbar_arrive(bar_addr(s.o_empty));
        const float ls = transpose_reduce<CW, false>(lsum);
        if (lane < CW) red[wiw * 32 + lane] = ls;
        if (!group_sync(grp, s.abort, gph)) goto out;
        SSD_TRACE(if (tid == 0 && jl < kTraceItems) TE[jl * 4 + 2] = (unsigned)(clock64() - clk0));
        // Each thread sums the four warps' partial row sums itself (all shared reads before the global
        // stores): no second group barrier.  The next write to red comes after the next item's first
        // vote barrier.
        float inv[CW];
#pragma unroll
        for (int j = 0; j < CW; j += 4) {
          float4 l4 = *reinterpret_cast<const float4 *>(red + j);
#pragma unroll
          for (int w = 1; w < 4; ++w) {
            const float4 p = *reinterpret_cast<const float4 *>(red + w * 32 + j);
            l4.x += p.x; l4.y += p.y; l4.z += p.z; l4.w += p.w;
          }
          inv[j] = l4.x; inv[j + 1] = l4.y; inv[j + 2] = l4.z; inv[j + 3] = l4.w;
        }
        const int64_t prow = ((int64_t)u * a.S_max + it.split) * R;
        if (tw < CW) {
          const int r = c0 + tw;
          if (r < R) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) l += red[w * 32 + tw];
            a.lse_parts[prow + r] = l > 0.f ? (s.mref[r] + __log2f(l)) * kLn2 : -INFINITY;
          }
          s.mref[r] = r < R ? -INFINITY : INFINITY;  // the next item's starting reference
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) inv[j] = inv[j] > 0.f ? __fdividef(1.f, inv[j]) : 0.f;
#pragma unroll
        for (int j = 0; j < CW; ++j)
          if (c0 + j < R) a.o_parts[(prow + c0 + j) * 128 + tw] = o[j] * inv[j];
      }
      SSD_TRACE(if (tid == 0 && jl < kTraceItems) {
        TE[jl * 4 + 3] = (unsigned)(clock64() - clk0);
        TR[6 + 3 * jl] = clock64() - clk0;
        TR[3] = jl + 1;
      });
      item = next_item;
      it = nx;
    }
  out:;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  SSD_TRACE(if (tid == 0) {
    TR[2] = global_ns();
    TR[127] = clock64() - clk0;
  });
  if (tid == 0 && *reinterpret_cast<volatile int *>(s.abort)) atomicOr(a.status, (unsigned)SSD_FAULT_TIMEOUT);
  if (warp == kTcMmaWarp) tmem_dealloc(tm, C::TMEM_COLS);
  // The last block to finish returns the item counter and the finished count to zero for the next
  // call (the counter area's contract).  Every block's draws completed before its count.
  if (tid == 0 && atomicAdd(a.sched + 1, 1) == (int)gridDim.x - 1) {
    __threadfence();
    atomicExch(a.sched, 0);
    atomicExch(a.sched + 1, 0);
  }
}

// ------------------------------------------------------------------------------------------------
// Host side.
// ------------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

bool verify_tc_supported(const ssd_paged_kv *kv, int R) {
  // max_seq_len below 2^24 keeps a unit's split count within the 16 bits the item decode stores it in.
  return kv->dtype == SSD_DTYPE_BF16 && kv->d == 128 && kv->page_size >= 8 && R <= 64 && kv->batch <= kTcMaxBatch &&
         kv->max_seq_len < (1 << 24) && (int64_t)kv->num_pages * 2 * kv->h_kv * kv->page_size < (1ll << 31);
}

template <int NP>
static int launch_tc(const CUtensorMap &map, const CUtensorMap &qmap, const VerifyArgs &a, int box_rows, int grid,
                     cudaStream_t st) {
  constexpr int smem = TcCfg<NP>::SMEM;
  int rc = ensure_smem<verify_tc_kernel<NP>>(smem);
  if (rc) return rc;
  return launch(verify_tc_kernel<NP>, dim3(grid), dim3(kTcThreads), smem, st, "verify_tc_kernel", map, qmap, a,
                box_rows);
}

int launch_verify_tc(const ssd_paged_kv *kv, const VerifyArgs &a, cudaStream_t st, int max_blocks) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(SSD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const int box_rows = kv->page_size < kTcTile ? kv->page_size : kTcTile;
  // The pool's 256-byte K / V rows as (64 columns, row in an 8-row group, 64-column panel, 8-row group):
  // one box takes box_rows rows of both panels and lands as [group][panel][8 rows x 128 B].
  CUtensorMap map;
  cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)kv->num_pages * 2 * kv->h_kv * kv->page_size / 8};
  cuuint64_t strides[3] = {256, 128, 2048};
  cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)box_rows / 8};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(kv->pool), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SSD_ERR_CUDA, "cuTensorMapEncodeTiled (KV pool) failed (%d)", (int)r);
  // Queries [B][n_c][h_q][128] as (64-column panel, panel, head, request*candidate); one box holds the
  // G heads x n_c candidates of a (request, KV head) for one panel.
  CUtensorMap qmap;
  cuuint64_t qdims[4] = {64, 2, (cuuint64_t)a.h_q, (cuuint64_t)kv->batch * a.n_c};
  cuuint64_t qstrides[3] = {128, 256, (cuuint64_t)a.h_q * 256};
  cuuint32_t qbox[4] = {64, 1, (cuuint32_t)a.G, (cuuint32_t)a.n_c};
  cuuint32_t qes[4] = {1, 1, 1, 1};
  r = enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(a.q), qdims, qstrides, qbox, qes,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SSD_ERR_CUDA, "cuTensorMapEncodeTiled (queries) failed (%d)", (int)r);
  const int64_t items_max = (int64_t)kv->batch * kv->h_kv * a.S_max;
  int grid = (int)(items_max < sm_count() ? items_max : sm_count());
  if (max_blocks > 0 && grid > max_blocks) grid = max_blocks;
  if (grid <= 0) return SSD_OK;
  if (!a.sched) return fail(SSD_ERR_INVALID_ARG, "verify_tc_kernel: no item counter");
  return a.R <= 32 ? launch_tc<32>(map, qmap, a, box_rows, grid, st) : launch_tc<64>(map, qmap, a, box_rows, grid, st);
}

}  // namespace ssd

#ifdef SSD_VERIFY_TRACE
// Diagnostic build only: copies the timeline record (kTraceBlocks x kTraceSlots 64-bit words) of the
// last verify launch to host memory.
extern "C" int ssd_verify_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
// Diagnostic build only: the softmax stage record (kTraceBlocks x kTraceStage x 8 32-bit words).
extern "C" int ssd_verify_stage_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_stage_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_stage_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
// Diagnostic build only: the producer's item-start record (kTraceBlocks x kTraceItems x 4 words).
extern "C" int ssd_verify_prod_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_prod_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_prod_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
// Diagnostic build only: the epilogue record (kTraceBlocks x kTraceItems x 4 32-bit words).
extern "C" int ssd_verify_epi_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_epi_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_epi_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
// Diagnostic build only: the masked-tile record (kTraceBlocks x kTraceMasked x 8 32-bit words).
extern "C" int ssd_verify_masked_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_masked_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_masked_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
// Diagnostic build only: the per-tile record (kTraceBlocks x kTraceTiles x kTT 32-bit words).
extern "C" int ssd_verify_tile_trace(void *dst, size_t bytes) {
  if (!dst || bytes > sizeof(ssd::g_verify_tile_trace)) return SSD_ERR_INVALID_ARG;
  return cudaMemcpyFromSymbol(dst, ssd::g_verify_tile_trace, bytes) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
#endif
