/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DSA indexer decode library.
 *
 * The library scores a paged FP8 index-K cache against FP8 queries (paged MQA
 * logits), bins every live score into a 1024-bin coarse histogram inside the
 * same kernel, selects the exact top-k columns per row from that histogram,
 * and builds the two-level candidate path (block maxima over 8-score blocks,
 * block top-k, an ascending padded block table, sparse logits over the chosen
 * blocks, and a top-k over FP16 scores).
 *
 * Sources, cited by page title and section:
 *   [DG94]   DeepGEMM PR #94 "[SM100] Paged MQA logits: fused coarse score
 *            histogram for LiteTopK decode" -- "What this adds", "Producer
 *            cost", commit 2d3b1c1, cross-referenced SGLang commit 7e252c5.
 *   [SG38944] SGLang PR #38944 "[DSV4.1] Enable the two-level candidate indexer
 *            on DeepGEMM's paged sparse MQA logits" -- squashed commit texts,
 *            "What this enables", "Structure", "Tests".
 *   [VL52696] vLLM PR #52696 "[Performance][MLA] Use FP16 logits for sparse
 *            indexer" -- "Summary", "Why".
 *
 * Conventions for every entry point:
 *   - Data pointers are DEVICE pointers owned by the caller unless a comment
 *     says otherwise; the library never frees or retains them past the call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The library allocates no device memory: scratch space comes
 *     from a caller-owned workspace sized by dsa_workspace_size().  The one
 *     exception is dsa_coarse_hist_topk_noalloc, whose scratch is a static
 *     device array of the library (about 5.3 MB per GPU that loads it).
 *   - Host-side argument checks run before anything is launched and return a
 *     status synchronously; nothing is launched when the status is not DSA_OK.
 *   - Problems only the device can see (a page id outside the pool, a context
 *     length beyond the page table or the output stride, a wait that ran out)
 *     are recorded as bits in the workspace's device status word and the
 *     kernel skips or clamps the offending access; they never trap.  Read the
 *     word with dsa_read_device_status().
 *   - Row r = b * next_n + j belongs to request b; it sees
 *     n_r = context_lens[b] - (next_n - 1 - j) keys ("token j of a request
 *     sees L + j keys", [DG94] "Producer cost", with context_lens[b] = L +
 *     next_n - 1).
 *   - Supported shapes follow [DG94] "What this adds": H = 32 heads, D = 128,
 *     FP8 E4M3 q and K, FP32 kscale, weights and logits, next_n in 1..4,
 *     page size 64 or 128 ([SG38944]: the metadata builder takes 64 or 128).
 *     Anything else returns DSA_ERR_UNSUPPORTED.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes returned by every entry point ------------------------- */
typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* NULL pointer, negative size, bad stride        */
  DSA_ERR_UNSUPPORTED = 2,   /* shape outside the supported set                */
  DSA_ERR_MISALIGNED = 3,    /* pointer or stride breaks an alignment rule     */
  DSA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed              */
  DSA_ERR_WORKSPACE = 5      /* workspace NULL or smaller than required        */
} dsa_status_t;

/* ---- device status word bits (sticky; see dsa_read_device_status) ------- */
#define DSA_DEV_TIMEOUT 0x1u  /* a bounded wait in a kernel ran out; the kernel
                                 drained its copies and returned early        */
#define DSA_DEV_BOUNDS 0x2u   /* a page id outside [0, num_pages), a context
                                 length beyond page_table_stride * page_size or
                                 the output stride, or a block id beyond the
                                 row; the access was skipped or clamped        */

#define DSA_NUM_BINS 1024     /* coarse histogram bins per row ([DG94])        */
#define DSA_MAX_TOPK 2048     /* largest k of the selects                      */
#define DSA_CAND_CAP 8192     /* threshold-bin candidates kept per row, the
                                 default capacity of FusedDecodePlan ([DG94],
                                 SGLang commit 7e252c5)                        */
#define DSA_OUT_F32 0
#define DSA_OUT_F16 1
#define DSA_OUT_BF16 2

/* Human-readable name of a dsa_status_t (static storage). */
const char *dsa_status_string(int32_t status);

/* Last CUDA error code seen by the library in this thread (0 if none). */
int32_t dsa_last_cuda_error(void);

/* Library version, as an integer major*10000 + minor*100 + patch. */
int32_t dsa_version(void);

/* ---- workspace ----------------------------------------------------------
 * One caller-owned device buffer serves every entry point.  It holds the
 * device status word, per-row select counters, the threshold-bin candidate
 * buffer (DSA_CAND_CAP entries per row), a histogram for selects that are not
 * given one, and a 4096-bin fine histogram per row for a threshold bin that
 * holds more than DSA_CAND_CAP scores (about 86 KiB per row in all).
 * `max_rows` is the largest row count any call will use.  The buffer must be
 * zero-filled once before first use (dsa_workspace_init);
 * every completed call leaves its counters at zero again, so no per-call
 * clearing is needed.  Calls that share a workspace must be ordered on one
 * stream (or otherwise serialised): concurrent calls on one workspace race. */
size_t dsa_workspace_size(int32_t max_rows);

/* Zero-fill the workspace on `stream` (also clears the device status word). */
int32_t dsa_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/* Copy the device status word to *out_host (synchronises `stream`). */
int32_t dsa_read_device_status(const void *workspace, void *stream, uint32_t *out_host);

/* ---- paged MQA logits with the fused coarse histogram -------------------
 * [DG94] "What this adds" and the indexer logits formula:
 *   logits[r, t] = sum_h weights[r, h] * ReLU( (sum_d q[r, h, d] * k[t, d]) * kscale[t] )
 * for every live column t < n_r; dead columns are not written.  K token t of
 * request b is read from physical slot s = page_table[b * page_table_stride +
 * t / page_size] * page_size + t % page_size.
 *
 *   q            [B*next_n][num_heads][head_dim] FP8 E4M3 bytes, 16-byte aligned
 *   kv_pages     [num_pages][page_size][head_dim] FP8 E4M3 bytes, 16-byte aligned
 *   kscale       [num_pages][page_size] float, 16-byte aligned
 *   weights      [B*next_n][num_heads] float, 16-byte aligned
 *   page_table   [B][page_table_stride] int32 physical page ids
 *   context_lens [B] int32
 *   logits       [B*next_n][logits_stride] float
 *   histogram    NULL, or [B*next_n][1024] int32, 8-byte aligned: every live,
 *                non-NaN score adds 1 to bin(score) of its row.  Counts are
 *                ADDED to what is there (zero it before the first call; the
 *                consumer resets it -- see dsa_coarse_hist_topk).  Bins
 *                descend: bin 0 holds the largest scores; |x| < 16 uses the
 *                FP16-RN exponent and 4 mantissa bits, 16 <= |x| < 223 unit
 *                bins, |x| >= 223 one saturating bin at each end.
 *   amax         NULL, or [B*next_n][amax_stride] float: the block maxima of
 *                dsa_block_amax8 computed in the same pass ([SG38944]
 *                amax8_varlen), bitwise equal to that entry point's output;
 *                rows with at most amax_skip_if_blocks_le blocks are skipped
 *                when that is > 0.
 * With or without the histogram and block maxima the logits are bitwise
 * identical. */
int32_t dsa_paged_mqa_logits(const uint8_t *q, const uint8_t *kv_pages, const float *kscale,
                             const float *weights, const int32_t *page_table,
                             int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                             int32_t next_n, int32_t num_heads, int32_t head_dim,
                             int32_t page_size, int32_t num_pages, float *logits,
                             int64_t logits_stride, int32_t *histogram, float *amax,
                             int64_t amax_stride, int32_t amax_skip_if_blocks_le,
                             void *workspace, size_t ws_bytes, void *stream);

/* ---- paged MQA logits over an MXFP4 index-K cache ------------------------
 * The next index-key format the pages point to: [SG38944] (Hopper prefill
 * commit text: block-scaled E2M1 index keys decoded to E4M3) and [VL52696]
 * ("Why"; the MXFP4 indexer-cache tests with a packed 68-byte layout).  Per
 * token: 128 E2M1 codes packed two per byte, dimension 2i in the low nibble
 * of byte i (64 bytes), and 4 UE8M0 block exponents, exponent j covering
 * dimensions 32j .. 32j+31 (4 bytes); k[d] = E2M1(code) * 2^(e[d / 32] - 127)
 * and no per-token kscale.  The logits are those of dsa_paged_mqa_logits
 * with that key and kscale = 1:
 *   logits[r][t] = sum_h w[r][h] * ReLU(q[r][h] . k[t])  for t < n_r,
 * computed on the block-scaled tensor-core MMA (E2M1 x E4M3, the exponents
 * applied per 32-dimension block as scale factors).
 *   k_codes  [num_pages][page_size][64] uint8, 32-byte aligned
 *   k_exp    [num_pages][page_size][4] uint8, 16-byte aligned
 * Every other argument, layout, the fused histogram and the error behaviour
 * are those of dsa_paged_mqa_logits (no block-maxima output).  The pages
 * restrict their fused histogram to FP8 keys; here the histogram is taken in
 * the same epilogue for either key format. */
int32_t dsa_paged_mqa_logits_mx(const uint8_t *q, const uint8_t *k_codes, const uint8_t *k_exp,
                                const float *weights, const int32_t *page_table,
                                int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                                int32_t next_n, int32_t num_heads, int32_t head_dim,
                                int32_t page_size, int32_t num_pages, float *logits,
                                int64_t logits_stride, int32_t *histogram, void *workspace,
                                size_t ws_bytes, void *stream);

/* ---- histogram-driven exact top-k ---------------------------------------
 * SGLang commit 7e252c5 (select.cuh, cross-referenced from [DG94]): per row,
 * find the threshold bin T from the coarse histogram (the bins above T hold
 * fewer than k scores, T completes k), emit every score in a bin above T,
 * collect the scores of bin T (at most DSA_CAND_CAP) and refine them exactly.
 * When the histogram shows bin T holding more than DSA_CAND_CAP scores, the
 * pass builds a 4096-bin fine histogram of bin T instead and a second pass
 * collects inside its threshold fine bin.  A histogram that does not match
 * the row (stale), or a fine bin still over capacity, falls back to an exact
 * whole-row radix select instead of raising a device error.
 * Rows of at most 131072 scores (stride <= 131072) take one launch: a cluster
 * of eight CTAs per row reads the row once into shared memory; it builds the
 * fine histogram whenever bin T holds more than 512 scores, so at most 512
 * candidates are usually left to rank.  Longer rows take the multi-CTA passes.
 *
 * Rows: r in [0, R); row r has n_r = ceil_div(context_lens[r / next_n] -
 * (next_n - 1 - r % next_n), len_div) live scores (len_div = 1 for logits
 * rows, 8 for rows of block maxima).
 *   logits       [R][stride] float; dead columns are never read
 *   histogram    [R][1024] int32 built by dsa_paged_mqa_logits for these rows,
 *                or NULL: the library builds it in the workspace first
 *   reset_histogram  nonzero: zero the caller's histogram rows after use (the
 *                consumer reset the histogram contract asks for)
 *   out_idx      [R][k] int32: the k columns with the largest scores, ties
 *                to the lower column, NaN never selected; order within a row
 *                is unspecified; rows with fewer than k live non-NaN scores
 *                are padded with -1
 *   fallback_flags NULL or [R] int32: 0 = histogram path (with or without
 *                the fine pass), 1 = stale histogram, 2 = threshold bin over
 *                capacity even after the fine pass
 * k <= DSA_MAX_TOPK. */
int32_t dsa_coarse_hist_topk(const float *logits, int64_t stride, const int32_t *context_lens,
                             int32_t next_n, int32_t len_div, int32_t R, int32_t *histogram,
                             int32_t reset_histogram, int32_t k, int32_t *out_idx,
                             int32_t *fallback_flags, void *workspace, size_t ws_bytes,
                             void *stream);

/* Kernel launches one dsa_coarse_hist_topk call makes on rows of `stride`
 * scores, with (has_histogram != 0) or without a caller histogram: 1 when
 * stride <= 131072 (one cluster of eight CTAs per row, the row kept in their
 * shared memory), else 2 with a histogram (pass, refine pass) and 3 without
 * (histogram build first).  Host only, no device work; -DSA_ERR_INVALID_ARG
 * for stride < 1. */
int32_t dsa_coarse_hist_topk_launches(int64_t stride, int32_t has_histogram);

/* ---- several top-k problems in one launch --------------------------------
 * Not a separate operation of the source pages: the decode step's top-2048 of
 * the logits rows and top-kb of the block-maxima rows ([SG38944]) are
 * independent, so they can share one launch.  Each problem has exactly the
 * arguments and results of dsa_coarse_hist_topk; no two problems may write
 * the same memory.  One workspace serves all of them: it must be sized for
 * the sum of their R (problem i uses the rows after those of problems
 * 0..i-1).  When count <= DSA_TOPK_BATCH_MAX and every stride is at most
 * 131072 the problems run in one launch, otherwise one after another on the
 * stream.  Problems with R = 0 are skipped unchecked (their pointers may be
 * NULL); argument errors are reported for the first offending problem before
 * anything is launched.
 *
 * Block output (block_k > 0, rows of scores: len_div = 1, stride <= 131072):
 * the same launch also selects, per row, the block_k blocks of 8 consecutive
 * scores with the largest block maxima -- exactly what dsa_block_amax8 (no
 * skipped rows) followed by dsa_coarse_hist_topk with len_div = 8 and k =
 * block_k returns ([SG38944] amax8_varlen + top-kb over the maxima): the
 * maximum ignores NaN scores, a block of NaN only is never selected, the
 * newest block (the one holding the row's last live score) counts as +inf,
 * ties go to the lower block.  The maxima are taken from the scores the
 * select already holds, never written to memory.  No histogram of the
 * maxima is needed: every block whose maximum lies above the score select's
 * emit threshold holds an emitted score, so when at least block_k blocks
 * (the newest one included) lie above it, the top block_k are selected
 * exactly among those (at most k of them); otherwise the exact select runs
 * over every block maximum of the row.
 *   block_out_idx         [R][block_k] int32 block ids, -1 padded, any order
 *   block_fallback_flags  NULL or [R] int32: 0, or 2 when more blocks lay
 *                         above the threshold than k (an inconsistent
 *                         histogram) and the whole-row select ran */
#define DSA_TOPK_BATCH_MAX 4
typedef struct dsa_topk_problem {
  const float *logits;
  int64_t stride;
  const int32_t *context_lens;
  int32_t *histogram;
  int32_t *out_idx;
  int32_t *fallback_flags;
  int32_t *block_out_idx;         /* NULL unless block_k > 0 */
  int32_t *block_fallback_flags;  /* NULL or [R] */
  int32_t next_n;
  int32_t len_div;
  int32_t R;
  int32_t reset_histogram;
  int32_t k;
  int32_t block_k;                /* 0: no block output */
  /* NULL, or the block output becomes the sorted block table of
   * [SG38944] sort_candidate_blocks in the same launch: exactly what
   * dsa_sort_candidate_blocks (row_to_req NULL, next_n as above) writes for
   * these block ids -- ascending, INT32_MAX padded, the identity table for
   * rows of at most block_k blocks -- with its physical blocks and live
   * lengths (either may be NULL) */
  const int32_t *block_page_table;  /* [B][block_page_table_stride] */
  int64_t block_page_table_stride;
  int32_t block_page_size;          /* 64 or 128 */
  int32_t *block_phys;              /* NULL or [R][block_k] */
  int32_t *block_valid_lens;        /* NULL or [R] */
} dsa_topk_problem;

int32_t dsa_coarse_hist_topk_batch(const dsa_topk_problem *problems, int32_t count,
                                   void *workspace, size_t ws_bytes, void *stream);

/* Kernel launches dsa_coarse_hist_topk_batch makes for these problems (host
 * only, no device work); -DSA_ERR_INVALID_ARG for a bad count or stride. */
int32_t dsa_coarse_hist_topk_batch_launches(const dsa_topk_problem *problems, int32_t count);

/* ---- top-k without a caller workspace --------------------------------------
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory at the point where they select -- for
 * example code running inside a framework that owns every allocation, or a
 * host callback that must not call cudaMalloc -- and so cannot provide the
 * workspace dsa_coarse_hist_topk needs.
 *
 * Same arguments, results and fallbacks as dsa_coarse_hist_topk, minus the
 * workspace: the scratch (counters, candidates, histograms) lives in one
 * static device array inside the library, sized for DSA_NOALLOC_MAX_ROWS rows
 * (about 5.3 MB, held on every GPU that loads the library until the process
 * exits).  R > DSA_NOALLOC_MAX_ROWS returns DSA_ERR_UNSUPPORTED.  The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make this first call
 *     before any stream capture.
 *   - Every call shares the one array and clears the parts that must start at
 *     zero itself (the kernels leave them at zero too, but a call that did
 *     not run to the end would otherwise leave them dirty for the next).  Calls whose kernels overlap on the GPU (other streams,
 *     other host threads) race on it and give wrong results: serialise them.
 *   - Device-side anomaly bits of this variant stay in the library's array and
 *     are not reported; fallback_flags still reports per-row fallbacks. */
#define DSA_NOALLOC_MAX_ROWS 64
int32_t dsa_coarse_hist_topk_noalloc(const float *logits, int64_t stride,
                                     const int32_t *context_lens, int32_t next_n,
                                     int32_t len_div, int32_t R, int32_t *histogram,
                                     int32_t reset_histogram, int32_t k, int32_t *out_idx,
                                     int32_t *fallback_flags, void *stream);

/* ---- block maxima over 8-score blocks ------------------------------------
 * [SG38944] amax8_varlen: for row r with n_r live scores and
 * nb = ceil(n_r / 8) blocks, amax[r][i] = max(logits[r][8i .. 8i+7]) for
 * i < nb - 1 (NaN ignored; an all-NaN block stays NaN), amax[r][nb-1] = +inf
 * (the newest block is always chosen), nothing written past nb.  Rows with
 * nb <= skip_if_blocks_le are skipped when skip_if_blocks_le > 0 (their block
 * table is the identity anyway).
 *   logits [R][stride] float, 16-byte aligned, stride % 4 == 0
 *   amax   [R][amax_stride] float */
int32_t dsa_block_amax8(const float *logits, int64_t stride, const int32_t *context_lens,
                        int32_t next_n, int32_t R, int32_t skip_if_blocks_le, float *amax,
                        int64_t amax_stride, void *workspace, size_t ws_bytes, void *stream);

/* ---- candidate block table ----------------------------------------------
 * [SG38944] sort_candidate_blocks: in place, the selected block ids of each
 * row (any order, -1 padded) become the ascending INT32_MAX-padded table that
 * the sparse logits read; rows with nb <= kb get the identity table
 * 0 .. nb-1.  Also emits, when the pointers are not NULL:
 *   phys_blocks [R][kb]: the same blocks as pool slot / 8 through the row's
 *               page table (INT32_MAX for padding; needs page_size % 8 == 0)
 *   valid_lens  [R]: live tokens covered by the table ([SG38944]
 *               candidate_row_lens); the live positions form a prefix of the
 *               sparse row because the newest (possibly partial) block has the
 *               largest id.
 * Row r uses page-table row r / next_n.  Ids outside [0, nb) are dropped and
 * flagged DSA_DEV_BOUNDS.  kb <= 4096. */
int32_t dsa_sort_candidate_blocks(int32_t *block_ids, int32_t kb, const int32_t *context_lens,
                                  int32_t next_n, int32_t R, const int32_t *page_table,
                                  int64_t page_table_stride, int32_t page_size,
                                  int32_t *phys_blocks, int32_t *valid_lens, void *workspace,
                                  size_t ws_bytes, void *stream);

/* ---- sparse MQA logits over the chosen blocks ----------------------------
 * [SG38944] "What this enables" (fp8_fp4_paged_sparse_mqa_logits scores only
 * the published blocks): position i < kb*8 of row r is token
 * t = block_table[r][i / 8] * 8 + i % 8 and gets the paged MQA logit of
 * (r, t) -- bitwise equal to dsa_paged_mqa_logits at (r, t) -- or -inf when
 * the table entry is padding (INT32_MAX) or t >= n_r.  Inputs as for
 * dsa_paged_mqa_logits; kb % 16 == 0.
 *   out        [R][out_stride] float (DSA_OUT_F32) or FP16 bits (DSA_OUT_F16,
 *              round-to-nearest-even of the float logit, [VL52696] "Why":
 *              the logits kernel writes FP16 directly) or BF16 bits
 *              (DSA_OUT_BF16, round-to-nearest-even, the BF16 sibling),
 *              out_stride >= kb*8
 *   phys_blocks, valid_lens  both NULL, or both the outputs of
 *              dsa_sort_candidate_blocks for this table: the K rows are then
 *              read straight from the physical blocks (no page-table read
 *              per block) and position i is live iff i < valid_lens[r] (the
 *              table's live positions form a prefix); same results. */
int32_t dsa_sparse_mqa_logits(const uint8_t *q, const uint8_t *kv_pages, const float *kscale,
                              const float *weights, const int32_t *page_table,
                              int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                              int32_t next_n, int32_t num_heads, int32_t head_dim,
                              int32_t page_size, int32_t num_pages, const int32_t *block_table,
                              int32_t kb, const int32_t *phys_blocks, const int32_t *valid_lens,
                              void *out, int32_t out_dtype, int64_t out_stride, void *workspace,
                              size_t ws_bytes, void *stream);

/* ---- row pairing of the sparse pass ---------------------------------------
 * [SG38944] commit text on DeepGEMM's sparse schedule: two consecutive rows
 * of one request share one KV pass, each keeping its own block list and
 * output layout (the rows share their page-table row).  Units: within each
 * request, rows 2m and 2m+1 form unit b * ceil(next_n / 2) + m; an odd last
 * row is a unit of its own.  U = B * ceil(next_n / 2) = dsa_pair_units().
 *
 * dsa_sort_candidate_blocks_paired: everything dsa_sort_candidate_blocks
 * does for the B * next_n rows (the same tables, physical blocks and live
 * lengths, bit for bit; valid_lens is required here), in one launch of U
 * CTAs, plus per unit the ascending union of its rows' tables:
 *   union_phys [U][2*kb]  physical block of union entry e (pool slot / 8),
 *                         INT32_MAX past the union
 *   union_pos  [U][2*kb]  (pos_a + 1) | (pos_b + 1) << 16: the entry's position
 *                         in each row's table, 0 where the row does not hold
 *                         the block; 0 past the union
 *   union_len  [U]        entries in the union
 * All caller-owned device buffers; kb <= 4096; page_size % 8 == 0. */
int32_t dsa_pair_units(int32_t B, int32_t next_n);
int32_t dsa_sort_candidate_blocks_paired(int32_t *block_ids, int32_t kb,
                                         const int32_t *context_lens, int32_t next_n, int32_t B,
                                         const int32_t *page_table, int64_t page_table_stride,
                                         int32_t page_size, int32_t *phys_blocks,
                                         int32_t *valid_lens, int32_t *union_phys,
                                         int32_t *union_pos, int32_t *union_len,
                                         void *workspace, size_t ws_bytes, void *stream);

/* dsa_sparse_mqa_logits_paired: the same output as dsa_sparse_mqa_logits
 * with phys_blocks and valid_lens (bitwise), computed per unit: each union
 * entry's K rows are read once and scored for both rows of the unit in one
 * tcgen05 MMA with N = 64 (both rows' 32 heads); a row's score goes to its
 * own table position, and its positions past its table (padding) get -inf.
 * union_* and valid_lens come from dsa_sort_candidate_blocks_paired for the
 * same tables.  Other arguments as dsa_sparse_mqa_logits (kb % 16 == 0,
 * out_stride >= kb*8). */
int32_t dsa_sparse_mqa_logits_paired(const uint8_t *q, const uint8_t *kv_pages,
                                     const float *kscale, const float *weights,
                                     const int32_t *page_table, int64_t page_table_stride,
                                     const int32_t *context_lens, int32_t B, int32_t next_n,
                                     int32_t num_heads, int32_t head_dim, int32_t page_size,
                                     int32_t num_pages, int32_t kb, const int32_t *union_phys,
                                     const int32_t *union_pos, const int32_t *union_len,
                                     const int32_t *valid_lens, void *out, int32_t out_dtype,
                                     int64_t out_stride, void *workspace, size_t ws_bytes,
                                     void *stream);

/* ---- top-k over FP16 scores ---------------------------------------------
 * [VL52696] "Why": select on the packed FP16 score bits directly (both halves
 * of a 32-bit word are turned into order keys with one 32-bit operation), a
 * 10-bit coarse pass, then one exact refine pass over the remaining 6 key
 * bits.  Positions i < valid_lens[r] take part unless NaN; ties go to the
 * lower position (= lower column, the table being ascending).
 *   scores      [R][stride] uint16 FP16 bits, 4-byte aligned rows (stride even)
 *   block_table NULL: out_idx holds positions i; else [R][kb] and out_idx holds
 *               the logical column block_table[r][i/8]*8 + i%8 (the fused
 *               page-table transform of [SG38944] topk_bf16_small)
 *   out_idx     [R][k] int32, order unspecified, -1 padded
 * valid_lens[r] <= 16384, k <= DSA_MAX_TOPK. */
int32_t dsa_topk_fp16(const uint16_t *scores, int64_t stride, const int32_t *valid_lens,
                      int32_t R, int32_t k, const int32_t *block_table, int32_t kb,
                      int32_t *out_idx, void *workspace, size_t ws_bytes, void *stream);

/* The same select over BF16 scores (the BF16 sibling of the FP16 packed
 * select; [SG38944]'s topk_bf16_small with its fused page-table transform):
 * NaN (BF16 exponent field all ones, mantissa not 0) never selected, order by
 * the BF16 value, ties to the lower position; arguments as dsa_topk_fp16. */
int32_t dsa_topk_bf16(const uint16_t *scores, int64_t stride, const int32_t *valid_lens,
                      int32_t R, int32_t k, const int32_t *block_table, int32_t kb,
                      int32_t *out_idx, void *workspace, size_t ws_bytes, void *stream);

/* ---- one whole decode step ------------------------------------------------
 * The two-level step of [SG38944] "What this enables" / "Structure" with the
 * fused histogram of [DG94] "What this adds", as one host call: the dense
 * logits with the coarse histogram, then one select launch for the
 * top-k of every row, its top-kb blocks and their sorted table with physical
 * blocks and live lengths (the histogram cleared for the next step), the
 * sparse logits over those blocks in FP16, and the FP16 top-k with the table
 * transform -- exactly the calls dsa_paged_mqa_logits,
 * dsa_coarse_hist_topk_batch (block_k = kb, block_page_table given),
 * dsa_sparse_mqa_logits (DSA_OUT_F16) and dsa_topk_fp16 make, each with its
 * own argument checks, on one stream.  It spares a caller that launches
 * eagerly the per-call overhead of four bindings; the results are bitwise
 * those of the four calls.
 *   logits        [R][logits_stride] float, R = B * next_n; logits_stride at
 *                 most 131072 (longer rows: DSA_ERR_UNSUPPORTED -- make the
 *                 separate calls, whose select takes them in several launches)
 *   histogram     [R][1024] int32, zero on entry, cleared again by the select
 *   topk_idx      [R][k] top-k columns of the dense logits
 *   block_ids     [R][kb] the sorted block table; phys_blocks [R][kb];
 *                 valid_lens [R]
 *   sparse_scores [R][kb * 8] FP16 bits; sparse_idx [R][k] the top-k of the
 *                 sparse scores as logical columns
 * All buffers are the caller's; the workspace is sized for R rows.  Returns
 * the first failing call's status (the launches before it are queued). */
typedef struct dsa_decode_step_args {
  const uint8_t *q;
  const uint8_t *kv_pages;
  const float *kscale;
  const float *weights;
  const int32_t *page_table;
  int64_t page_table_stride;
  const int32_t *context_lens;
  int32_t B;
  int32_t next_n;
  int32_t page_size;
  int32_t num_pages;
  int32_t k;
  int32_t kb;
  float *logits;
  int64_t logits_stride;
  int32_t *histogram;
  int32_t *topk_idx;
  int32_t *block_ids;
  int32_t *phys_blocks;
  int32_t *valid_lens;
  uint16_t *sparse_scores;
  int32_t *sparse_idx;
} dsa_decode_step_args;

int32_t dsa_decode_step(const dsa_decode_step_args *args, void *workspace, size_t ws_bytes,
                        void *stream);

/* ---- diagnostics (same device functions as the kernels above) ------------
 * dsa_coarse_bins_range: out[i] = coarse bin of the float whose bit pattern is
 *   start + i (-1 for NaN), for i < count; out is int16 on the device.  Used
 *   to sweep all 2^32 patterns against an independent reference.
 * dsa_fp16_order_keys: out[i] = 16-bit order key of the FP16 pattern in[i]
 *   computed two halves per 32-bit word, as the FP16 select does (NaN -> 0);
 *   n even, both arrays device-resident.  dsa_bf16_order_keys: the same for
 *   BF16 patterns, as the BF16 select does.
 * dsa_wait_timeout_selftest: launches a kernel whose only wait is on a
 *   barrier nothing arrives on, bounded by `limit_cycles`; the kernel records
 *   DSA_DEV_TIMEOUT in the workspace status word and returns.
 * dsa_coarse_bin_key_ranges: out[2T], out[2T+1] = the lowest and highest
 *   FP32 order key (unsigned compare == value compare) of coarse bin T, for
 *   T = 0..1024 (T = 1024: an empty range, low > high), as the select kernel
 *   computes them in closed form; out is a device array of 2050 uint32. */
int32_t dsa_coarse_bins_range(uint32_t start, int64_t count, int16_t *out, void *stream);
int32_t dsa_coarse_bin_key_ranges(uint32_t *out, void *stream);
int32_t dsa_fp16_order_keys(const uint16_t *in, uint16_t *out, int64_t n, void *stream);
int32_t dsa_bf16_order_keys(const uint16_t *in, uint16_t *out, int64_t n, void *stream);
int32_t dsa_wait_timeout_selftest(uint64_t limit_cycles, void *workspace, size_t ws_bytes,
                                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
