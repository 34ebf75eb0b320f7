/*
 * ssd.h -- C ABI of libssd: GPU attention for sparse self-speculative decoding (sm_103a).
 *
 * One speculative round over a paged KV cache (SparseSpec, "Accelerating Large-Scale Reasoning
 * Model Inference: Self-Speculative Decoding with Sparse Attention", §4.1 PillarAttn, §2.3, §3.2):
 *   1. ssd_verify_attn  -- full attention of the k+1 candidate tokens of each request over its whole
 *                          cache, causal among the candidates; the same pass emits every KV token's
 *                          criticality (softmax probability summed over the query heads of the KV
 *                          group and the k+1 verify positions).
 *   2. ssd_select_topk  -- Top-K of the criticality per (request, KV head), ties to the lower index
 *                          (ssd_select_topp: the same with a per-row K from a top-p budget).
 *   3. ssd_draft_attn   -- the next k drafts: single-query attention over the selected tokens only
 *                          (ssd_draft_attn_packed: the first draft keeps the selected rows packed
 *                          for the others).
 * plus verify and select in one call (ssd_verify_select), the unified verify/draft call over a
 * mixed batch (§4.2 "fused attention"), the block-granular variant (SpecSA post, overlap-aware
 * grouped query execution; SparDA §2 max-pooling to a block grid), and around the round the KV
 * append / length rollback (SpecSA: accepted tokens' KV is kept, rejected ones' dropped) and the
 * phase assignment of the unified batch (§4.2).
 *
 * Conventions (all calls):
 *  - Every pointer argument named as "device" is device memory of the current CUDA device; host
 *    pointers are only the ssd_paged_kv struct itself and scalar outputs of ssd_status.
 *  - The caller owns all memory.  The library allocates nothing, keeps no pointer after a call
 *    returns, and takes scratch space only from the caller's workspace, sized by the matching
 *    ssd_*_workspace_bytes() query.  A workspace must be zero-filled once after allocation.  Its
 *    first 256 KiB hold only the library's counters, which every call returns to zero, so one
 *    workspace may then serve calls of any entry point and shape one after another.  It must not
 *    be shared by calls that may run concurrently.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    Argument errors are detected on the host and returned before anything is launched; launch
 *    failures return SSD_ERR_CUDA.  Data-dependent faults found on the device (a page id outside
 *    the pool, a token index >= its request's length, a length outside [0, max_seq_len], K > k_max)
 *    never trap: the offending load is skipped (zero-filled) and a bit is set in a device status
 *    word that ssd_status() reports.
 *  - The library never aborts, prints or traps.  ssd_last_error() returns a thread-local message
 *    for the last failing call on the calling thread.
 *  - Per device, the library keeps state for the life of the process: the device addresses of its
 *    status word and of ssd_draft_attn_static's built-in scratch, and its kernels' shared-memory
 *    limits.  After cudaDeviceReset (or any other teardown of a device's primary context) it must
 *    not be called on that device again in the same process.
 *  - SSD_FAULT_TIMEOUT means a copy or an MMA that a kernel waited for did not complete within
 *    about a second; the kernel stopped waiting, but the copy may still be in flight.  Treat the
 *    CUDA context as unusable after it.
 *  - Layouts are dense and row-major unless a stride argument says otherwise.
 *  - Notation: B requests, H_q query heads, H_kv KV heads, G = H_q / H_kv, d head dim (64 or 128),
 *    n_cand = k + 1, R = G * n_cand rows per (request, KV head) (R <= 64).  Query head h reads KV
 *    head h / G.  Request b holds L_b = seq_lens[b] tokens, its candidates at positions
 *    L_b - n_cand .. L_b - 1; candidate i sees tokens t <= L_b - n_cand + i.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssd_stream_t; /* == cudaStream_t */

enum ssd_status_code {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* null pointer, bad size or stride, inconsistent shapes */
  SSD_ERR_UNSUPPORTED = 2, /* dtype, head dim, page size or group shape outside what is built */
  SSD_ERR_WORKSPACE = 3,   /* workspace null or smaller than the query function says */
  SSD_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  SSD_ERR_TIMEOUT = 5      /* reserved, never returned: expired device waits raise SSD_FAULT_TIMEOUT */
};

enum ssd_dtype { SSD_DTYPE_F32 = 0, SSD_DTYPE_BF16 = 1 };

/* Device status word bits (ssd_status). */
enum ssd_device_fault {
  SSD_FAULT_PAGE = 1u,     /* a page id outside [0, num_pages) */
  SSD_FAULT_SEQLEN = 2u,   /* seq_lens[b] outside [0, max_seq_len] or shorter than n_cand */
  SSD_FAULT_INDEX = 4u,    /* a draft index outside [0, L_b) */
  SSD_FAULT_KMAX = 8u,     /* a requested K larger than k_max (output truncated to k_max) */
  SSD_FAULT_UNION = 16u,   /* a block union larger than umax (output truncated) */
  SSD_FAULT_TIMEOUT = 32u, /* a bounded wait inside a kernel expired; that block's outputs are invalid */
  SSD_FAULT_VALUE = 64u    /* a score that must be >= 0 (top-p selection) was negative or NaN */
};

/*
 * Paged KV cache (SparseSpec §4.2: PagedAttention; a page of size 1 turns full attention into the
 * sparse token-list case, so both share one pipeline).
 *   pool        device, [num_pages][2][h_kv][page_size][d] of `dtype`; index 0 = K, 1 = V.  Each
 *               (page, K|V, head) block of page_size * d elements is contiguous.  16-byte aligned.
 *   page_table  device int32 [batch][max_pages]: request b's token t lives in page
 *               page_table[b][t / page_size], slot t % page_size.  Entries past a request's last
 *               page are never read.
 *   seq_lens    device int32 [batch].
 *   max_seq_len host upper bound of seq_lens (sizes grids and workspaces);
 *               max_seq_len <= max_pages * page_size.
 */
typedef struct ssd_paged_kv {
  const void *pool;
  int dtype;
  int64_t num_pages;
  int page_size; /* power of two */
  int h_kv;
  int d; /* 64 or 128 */
  const int32_t *page_table;
  int max_pages;
  const int32_t *seq_lens;
  int batch;
  int max_seq_len;
} ssd_paged_kv;

/* Thread-local message describing the last failing call on this thread ("" if none). */
const char *ssd_last_error(void);

/* ABI version: (major << 16) | minor. */
int ssd_version(void);

/* Synchronises `stream`, then returns in *status the OR of all device fault bits raised by
 * kernels of this library on the current device since the previous ssd_status call, and clears
 * them.  Returns SSD_ERR_CUDA if the synchronisation reports an error. */
int ssd_status(ssd_stream_t stream, uint32_t *status);

/* ---------------------------------------------------------------------------------------------
 * Verify attention with fused criticality.
 * SparseSpec §4.1 (PillarAttn): the verify step runs full attention over the whole cache; its
 * kernel dumps the attention scores, caching logits and the log-sum-exp to rematerialise them;
 * the scores are reduced over the heads of a GQA group and the verify positions.  SpecAttn
 * (abstract): KV criticality is a byproduct of verification.
 *
 *   q        device [batch][n_cand][h_q][d] of kv->dtype (candidate i = verify position i).
 *   scale    softmax scale applied to q.k (typically 1/sqrt(d)); natural-base softmax.
 *   out      device float [batch][n_cand][h_q][d]: attention output.
 *   lse      device float [batch][n_cand][h_q] or NULL: natural-log log-sum-exp of the scaled logits.
 *   scores   device float [batch][h_kv][scores_stride] or NULL: scores[b][g][t] =
 *            sum over the G heads h of group g and candidates i of softmax_{b,h,i}(t) (0 where t is
 *            not visible to i).  Entries t >= L_b are not written.  scores_stride >= max_seq_len.
 *   bscores  device float [batch][h_kv][n_cand][bscores_stride] or NULL (block mode): for every
 *            candidate i, the per-candidate criticality sum over h of softmax_{b,h,i}(t) max-pooled
 *            over blocks of block_size tokens (block j = tokens [j*bs, min((j+1)*bs, L_b))).
 *            Blocks >= ceil(L_b / bs) are not written.  block_size must be 64 when bscores != NULL.
 *   workspace device, >= ssd_verify_workspace_bytes(kv, h_q, n_cand) bytes, 256-byte aligned.
 */
size_t ssd_verify_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand);
int ssd_verify_attn(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                    float *lse, float *scores, int64_t scores_stride, float *bscores,
                    int64_t bscores_stride, int block_size, void *workspace, size_t workspace_bytes,
                    ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Verify with the selection fused into its criticality pass (SparseSpec §4.1: Top-K is applied to
 * the scores the verify dumps; fusing removes the separate select launch and its read of the
 * scores).  Same arguments and results as ssd_verify_attn with scores (no block scores), plus the
 * Top-K that ssd_select_topk(scores, scores_stride, seq_lens, ks, batch, h_kv, 1, max_seq_len, idx,
 * k_max, cnt) would write: ks is device int32 [batch] (K per request), idx device int32
 * [batch][h_kv][k_max] (ascending, -1 padded), cnt device int32 [batch][h_kv]; K > k_max raises
 * SSD_FAULT_KMAX and keeps k_max.  The workspace is ssd_verify_workspace_bytes(kv, h_q, n_cand);
 * batch * h_kv must be at most 65534 (its counters share the workspace's counter area).
 */
int ssd_verify_select(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                      float *lse, float *scores, int64_t scores_stride, const int32_t *ks, int32_t *idx, int k_max,
                      int32_t *cnt, void *workspace, size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Top-K selection (SparseSpec §4.1: "Top-K on the dumped scores" gives the sparse pattern; §3.2,
 * §5.4: about 5% of the tokens).  Rows r = 0 .. n_groups*rows_per_group-1 of the score matrix
 * (device float, row stride `stride` elements) belong to group r / rows_per_group; row r has
 * n_r = ceil(lens[group] / len_div) entries and keeps K_r = min(ks[group], n_r) of them: the K_r
 * largest values, equal values broken toward the lower index.  idx (device int32 [rows][k_max])
 * receives the kept indices in ascending order, -1 padded; cnt (device int32 [rows]) receives K_r.
 * lens and ks are device int32 [n_groups].  max_len (host) bounds n_r.  Scores must not be NaN;
 * -0.0 ranks equal to +0.0.  Token level: rows_per_group = h_kv, lens = seq_lens, len_div = 1.
 */
int ssd_select_topk(const float *scores, int64_t stride, const int32_t *lens, const int32_t *ks,
                    int n_groups, int rows_per_group, int len_div, int max_len, int32_t *idx, int k_max,
                    int32_t *cnt, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Top-p selection: a per-row budget instead of a fixed K (SparseSpec §3.2 and §3.3 measure the
 * draft against "oracle top-k" attention and cite adaptive sparsity by hierarchical top-p pruning,
 * Twilight; §4.1: the selected set is the top of the verify scores).  Row r (same grouping, lengths and len_div as ssd_select_topk) keeps
 * K_r = min(K_p, k_max) entries, where K_p is the smallest count of the row's largest entries
 * (equal values toward the lower index) whose sum reaches p times the row's total; the kept set
 * is the Top-K_r set, written to idx / cnt exactly as ssd_select_topk writes it.  k_rows (device
 * int32 [rows]) receives K_r.  p is in [0, 1]; p = 0, an empty row or an all-zero row keeps
 * nothing.  Scores must be >= 0 (criticality is a sum of probabilities): a row holding a negative
 * value or NaN keeps nothing and raises SSD_FAULT_VALUE.  Sums are exact 64-bit fixed point in
 * units of 2^(ceil(log2 n_r) - 62) times the power of two just above the row's maximum; smaller
 * values round down to that unit.  Two kernels on `stream`: the counts, then the Top-K pass.
 */
int ssd_select_topp(const float *scores, int64_t stride, const int32_t *lens, float p, int n_groups,
                    int rows_per_group, int len_div, int max_len, int32_t *idx, int k_max, int32_t *cnt,
                    int32_t *k_rows, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Sparse draft attention (SparseSpec §4.1: each of the k drafts after a verify loads only the
 * selected tokens; §4.2: sparse attention is PagedAttention at page size 1).
 *   q    device [batch][h_q][d] of kv->dtype (one draft query per request).
 *   idx  device int32 [batch][h_kv][k_max], cnt device int32 [batch][h_kv]: the token list of
 *        each (request, KV head); each entry must be in [0, L_b).  Duplicates count twice.
 *   out  device float [batch][h_q][d]; lse device float [batch][h_q] or NULL.  An empty list
 *        gives out = 0 and lse = -inf.
 */
size_t ssd_draft_workspace_bytes(const ssd_paged_kv *kv, int h_q, int k_max);
int ssd_draft_attn(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                   const int32_t *cnt, float scale, float *out, float *lse, void *workspace,
                   size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Sparse draft attention with a row pack.  The k drafts of a round all attend the set the last
 * verify selected (SparseSpec §4.1: the pattern stays fixed until the next verify refreshes it), so
 * the first draft can leave the selected K and V rows in a contiguous buffer and the others read
 * them from there instead of through the index list and the page table.  Same arguments and
 * workspace as ssd_draft_attn, and the same results up to rounding: SSD_PACK_WRITE bit for bit;
 * SSD_PACK_READ of a bf16 cache runs one block per (request, KV head) with an online softmax over
 * the chunks, so its sums are taken in another order.  In addition:
 *   pack        device buffer of at least ssd_draft_pack_bytes(kv, k_max) bytes, 256-byte aligned,
 *               owned by the caller.  Its layout is private to the library.
 *   pack_mode   SSD_PACK_NONE: exactly ssd_draft_attn (pack unused, may be NULL).
 *               SSD_PACK_WRITE: ssd_draft_attn, and every selected row it read is stored in pack.
 *               SSD_PACK_READ: attends the rows the last SSD_PACK_WRITE call (or the last
 *               ssd_verify_select_packed call) on this pack stored;
 *               idx is not read (may be NULL) and the page table and lengths are not consulted, so
 *               no index or page fault is raised.  cnt and k_max must equal that call's and the
 *               selected tokens' K / V must be unchanged since (appending new tokens is fine); a cnt
 *               that grew reads rows the pack does not hold (wrong values, never outside pack).
 *               SSD_PACK_READ_DISCARD: SSD_PACK_READ, after which the pack's contents are undefined
 *               (for the last draft of a round: a bf16 pack's lines are dropped from the L2 cache
 *               without being written back to memory).  Write the pack again before the next read.
 * Entries of cnt outside [0, k_max] raise SSD_FAULT_KMAX in every mode.
 */
enum ssd_pack_mode { SSD_PACK_NONE = 0, SSD_PACK_WRITE = 1, SSD_PACK_READ = 2, SSD_PACK_READ_DISCARD = 3 };
size_t ssd_draft_pack_bytes(const ssd_paged_kv *kv, int k_max);
int ssd_draft_attn_packed(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                          const int32_t *cnt, float scale, float *out, float *lse, void *pack, size_t pack_bytes,
                          int pack_mode, void *workspace, size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * ssd_verify_select, and the selection's K and V rows stored in a row pack as an SSD_PACK_WRITE
 * draft over (idx, cnt, k_max) would store them, so that every draft of the round can read the pack
 * (SSD_PACK_READ) and none gathers through the index list (SparseSpec §4.1: the k drafts attend the
 * set this verify selects).  The selecting blocks know their unit's indices when they finish and
 * copy its rows then.  Same arguments and results as ssd_verify_select, plus:
 *   pack        device buffer of at least ssd_draft_pack_bytes(kv, k_max) bytes, 256-byte aligned,
 *               owned by the caller; its layout is private to the library.  A selected token whose
 *               page id is out of range stores zero rows (the verify raises SSD_FAULT_PAGE).
 *   pack_bytes  its size; smaller than needed: SSD_ERR_WORKSPACE.
 */
int ssd_verify_select_packed(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand, float scale, float *out,
                             float *lse, float *scores, int64_t scores_stride, const int32_t *ks, int32_t *idx,
                             int k_max, int32_t *cnt, void *pack, size_t pack_bytes, void *workspace,
                             size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * KV append and length advance (SpecSA post, "refresh/reuse NSA kernel fusion" and "branch
 * handling": the KV of accepted tokens is kept, that of rejected tokens dropped; SparseSpec §2.3: a
 * verify checks the k drafts plus one bonus position).  With this library's verify convention the
 * n_cand candidates of request b sit at positions L_b - n_cand .. L_b - 1, so a round is:
 *   ssd_kv_append(candidates' K/V) -> ssd_kv_advance(+n_cand) -> verify / select / drafts ->
 *   ssd_kv_advance(-(n_cand - accepted_b)).
 * The rejected candidates' rows stay in their pages past the request's end, where nothing reads them.
 *
 * ssd_kv_append: writes token j (0 <= j < n_new) of request b at position seq_lens[b] + j.
 *   k_new, v_new  device [batch][n_new][h_kv][d] of kv->dtype, 16-byte aligned.  kv->pool is written
 *                 (the struct's const qualifier notwithstanding); seq_lens is only read.
 *   The caller allocates the pages: page_table must map every new position.  A request whose new
 *   positions would pass max_seq_len (SSD_FAULT_SEQLEN) or use a page id outside the pool
 *   (SSD_FAULT_PAGE) is skipped as a whole; the others are written.
 * ssd_kv_advance: seq_lens[b] += delta[b] (device int32 arrays of `batch`); a result outside
 *   [0, max_seq_len] leaves seq_lens[b] unchanged and raises SSD_FAULT_SEQLEN.
 */
int ssd_kv_append(const ssd_paged_kv *kv, const void *k_new, const void *v_new, int n_new,
                  ssd_stream_t stream);
int ssd_kv_advance(int32_t *seq_lens, const int32_t *delta, int batch, int max_seq_len,
                   ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * ssd_draft_attn_static: ssd_draft_attn without a workspace.  The paper has no counterpart; this
 * is a library convenience.  It exists for callers that cannot allocate device memory where they
 * run the draft step: a plugin inside another runtime that owns all device allocations and passes
 * in only input and output buffers, or a serving loop that must not call cudaMalloc / cudaFree
 * (which can synchronise the whole device) while other streams are running.
 *
 * Same arguments, results and device-side fault reporting as ssd_draft_attn, minus workspace and
 * workspace_bytes.  The scratch is one built-in device array of SSD_DRAFT_STATIC_SCRATCH_BYTES
 * (16 MiB), held on every device that loads the library until the process exits.  The call
 * allocates and frees nothing.
 *  - A batch whose scratch does not fit returns SSD_ERR_WORKSPACE before anything is launched;
 *    use ssd_draft_attn for it.  The scratch is 4 bytes per (request, KV head) rounded up to 256,
 *    plus ssd_draft_workspace_bytes for the same arguments minus its 256 KiB counter area.
 *  - The first call on each device looks up the array's device address (with that device current)
 *    and keeps it; make that first call before any stream capture on the device.
 *  - Every call on a device uses the same array, which keeps the previous call's contents; the
 *    parts that must start at zero are cleared on `stream` before the kernel runs.  Calls whose
 *    work can overlap on the GPU (different streams with no ordering between them) race on the
 *    array and give wrong results: order them on one stream or with events.
 */
#define SSD_DRAFT_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
int ssd_draft_attn_static(const ssd_paged_kv *kv, const void *q, int h_q, const int32_t *idx, int k_max,
                          const int32_t *cnt, float scale, float *out, float *lse, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Unified launch (SparseSpec §4.2: requests of both phases in one batch; a persistent fused kernel
 * dispatches verify and draft work to their own tile code in one launch).  phase (device uint8
 * [batch]): 1 = verify, 0 = draft.  Verify-phase requests take q_verify/out_verify/lse_verify/
 * scores exactly as ssd_verify_attn; draft-phase requests take q_draft/idx/cnt/out_draft/lse_draft
 * exactly as ssd_draft_attn.  Rows of the other phase are left untouched.
 */
size_t ssd_unified_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand, int k_max);
int ssd_unified_attn(const ssd_paged_kv *kv, const uint8_t *phase, const void *q_verify,
                     const void *q_draft, int h_q, int n_cand, const int32_t *idx, int k_max,
                     const int32_t *cnt, float scale, float *out_verify, float *lse_verify,
                     float *scores, int64_t scores_stride, float *out_draft, float *lse_draft,
                     void *workspace, size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Phase assignment for the unified batch (SparseSpec §4.2, workload-aware scheduling: requests of
 * both phases are mixed evenly in every step; a greedy bin-packing keeps one bucket per phase and
 * gives each arriving request the least loaded one).  A bucket is a phase offset o in
 * [0, n_buckets) with n_buckets = k + 1: at step s a request with offset o is in phase
 * (s + o) mod n_buckets, where n_buckets - 1 is its verify and the other phases its k drafts.
 *
 * ssd_phase_assign (host only, no CUDA call): counts (host int32 [n_buckets], live requests per
 *   offset) is updated in place; offset_out (host int32 [n_new]) receives each arriving request's
 *   offset in arrival order: the bucket with the smallest count, ties to the lowest offset.  The
 *   caller decrements counts[o] when a request with offset o finishes.
 * ssd_phase_fill: phase (device uint8 [batch]) = 1 where request b verifies at `step`, 0 where it
 *   drafts -- the phase array of ssd_unified_attn.  offsets: device int32 [batch]; an offset
 *   outside [0, n_buckets) gives 0 and raises SSD_FAULT_INDEX.
 */
int ssd_phase_assign(int32_t *counts, int n_buckets, int n_new, int32_t *offset_out);
int ssd_phase_fill(const int32_t *offsets, int batch, int n_buckets, int64_t step, uint8_t *phase,
                   ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Block-granular variant (SpecSA post: overlap-aware grouped query execution -- candidates with
 * overlapping sparse layouts run together and share KV blocks; hierarchical layout management).
 *
 * ssd_block_union: for each unit u (= request * h_kv + KV head), the union of the n_cand
 * candidates' block lists blocks (device int32 [units][n_cand][kb], bcnt valid entries each, as
 * written by ssd_select_topk with rows_per_group = h_kv * n_cand) in ascending order: uidx (device
 * int32 [units][umax], -1 padded), umask (device uint32 [units][umax], bit i = candidate i chose the
 * block) and ucnt (device int32 [units]).  Block ids must be in [0, nblk_max); n_cand <= 32.
 *
 * ssd_block_sparse_attn: candidate i of request b attends to the tokens of its own blocks that
 * it can see (t < L_b and t <= L_b - n_cand + i); each union block is loaded once for all
 * candidates and heads of the unit.  q/out/lse as in ssd_verify_attn.  block_size must be 64.
 */
int ssd_block_union(const int32_t *blocks, const int32_t *bcnt, int n_units, int n_cand, int kb,
                    int nblk_max, int32_t *uidx, uint32_t *umask, int32_t *ucnt, int umax,
                    ssd_stream_t stream);
size_t ssd_block_sparse_workspace_bytes(const ssd_paged_kv *kv, int h_q, int n_cand, int umax);
int ssd_block_sparse_attn(const ssd_paged_kv *kv, const void *q, int h_q, int n_cand,
                          const int32_t *uidx, const uint32_t *umask, const int32_t *ucnt, int umax,
                          int block_size, float scale, float *out, float *lse, void *workspace,
                          size_t workspace_bytes, ssd_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Split-KV combine (the log-sum-exp merge the verify and draft passes use internally).
 * o_parts device float [n_rows][n_splits][d] (each split's normalised output), lse_parts device
 * float [n_rows][n_splits] (natural-log LSE of each split; -inf for an empty split).  Writes
 * out [n_rows][d] = sum_j exp(lse_j - lse*) o_j and lse [n_rows] = log sum_j exp(lse_j) (NULL to
 * skip); all-empty rows, and every row when n_splits = 0 (o_parts and lse_parts may then be NULL),
 * give out = 0, lse = -inf.
 */
int ssd_combine(const float *o_parts, const float *lse_parts, int n_rows, int n_splits, int d,
                float *out, float *lse, ssd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
