/*
 * gvr_topk.h -- C ABI of libgvrtopk: exact per-row top-K over fp32 sparse-attention indexer
 * scores by hint-free Guess-Verify-Refine (GVR) self-sampling, on one NVIDIA GB300 (sm_103a).
 *
 * The operation.  For every row r the library returns the K window-local indices of the K
 * largest scores of that row's valid window W_r = [a_r, a_r + nv_r) of
 * logits[r * row_stride + ...]:
 *   - "exact (tie-interchangeable) top-K": when several scores tie at the K-th largest value
 *     tau, any choice among the tied entries is correct; -0 and +0 are one tie class; +inf and
 *     -inf are ordinary values ("Block-skip fast path for self-sampling GVR top-K decode",
 *     TensorRT-LLM PR #18122, commit log "Contract" and "run_varlen");
 *   - a window with nv_r <= K yields the identity 0, 1, ..., nv_r - 1 followed by -1 pads
 *     ("Self-sampling GVR V2 prefill indexer top-K", PR #18702, section "Kernel");
 *   - the K indices of a longer row come in no particular order;
 *   - scores outside the window (padding, other requests, +inf/NaN/3e38/-inf poison) never
 *     influence the result; NaN inside a window is outside the contract: the result is then K
 *     distinct in-window indices, but which ones is unspecified.
 * How it is computed ("GVR K=2048 reg_clus with block64 sampling and parallel rescue",
 * PR #20998, sections "Why the GLM row overflows" and "What changes"): uniform block64
 * sampling of exactly K scores gives a value bracket [GMIN, GMAX]; a value histogram over the
 * bracket finds the bin that crosses tau; the members of that bin go to a bounded candidate
 * buffer and an exact refine picks the remaining winners; an invalid bracket or an overflowing
 * buffer sends the row to an exact radix rescue that runs on every CTA of the row's cluster.
 * Which kernel runs is decided on the host from row_stride, num_rows and the options alone: a
 * cluster of CTAs per row streaming the window through a shared-memory ring, or, for plain
 * calls with row_stride <= 16384 and at most four waves of rows, one CTA per row holding the
 * whole window in shared memory (GVR_FLAG_SHORT_KERNEL); the results are exact either way.
 *
 * Conventions shared by every entry point.
 *   - All pointers except `options` are DEVICE pointers into memory the caller owns.  The
 *     library allocates nothing, never reads device memory on the host and never
 *     synchronizes: each call validates its arguments on the host and enqueues ONE kernel on
 *     `stream` (a cudaStream_t; NULL is the legacy default stream).  The result is ready when
 *     the stream reaches that point.  The first call on a device sets kernel attributes once.
 *   - logits is fp32 [num_rows][row_stride], row-major with unit inner stride; its base must
 *     be 16-byte aligned and row_stride a multiple of 4 (float4 rows), 4 <= row_stride <
 *     2^31.  Reads stay inside each row's window, widened at its start only down to the
 *     16-byte boundary (never past the window's last score).
 *   - indices is int32 [num_rows][k] (row stride exactly k); values (when non-NULL) is fp32
 *     [num_rows][k].  Every one of the k slots of every row is written.
 *   - k must be 512, 1024 or 2048.
 *   - num_rows == 0 is a no-op that returns GVR_OK.
 *   - Errors are returned, never raised on the device: argument errors are detected on the
 *     host before anything is enqueued; GVR_ERR_LAUNCH is returned when cudaLaunchKernelEx
 *     returns an error for the one launch (no device, bad configuration, ...).
 *   - Device-side failure marker: every wait of the kernel for its staged scores is bounded
 *     (0.5 s).  A row whose wait gave up -- not expected to happen on a healthy GPU -- gets -2
 *     in every index slot instead of a selection (values are then unspecified).  -2 is never a
 *     valid index or pad: a caller that gathers with the indices must treat it as invalid.  The
 *     *_ex entry points also report it per row as GVR_PATH_DEVICE_ERROR in row_stats.
 *   - Calls may run concurrently on different streams: no state is shared between calls.
 */
#ifndef GVR_TOPK_H
#define GVR_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gvr_status {
  GVR_OK = 0,
  GVR_ERR_NULL = 1,   /* a required pointer is NULL */
  GVR_ERR_ALIGN = 2,  /* logits is not 16-byte aligned, or indices/values not 4-byte aligned */
  GVR_ERR_STRIDE = 3, /* row_stride is not a multiple of 4, below 4, or not below 2^31 */
  GVR_ERR_K = 4,      /* k is not 512, 1024 or 2048 */
  GVR_ERR_ARG = 5,    /* a negative row count, next_n < 1, compress_ratio < 1, bad options */
  GVR_ERR_LAUNCH = 6,   /* the kernel launch failed (no device, bad configuration, ...) */
  GVR_ERR_WORKSPACE = 7, /* the workspace is NULL, not 16-byte aligned or smaller than
                            gvr_workspace_size reports */
  GVR_ERR_NOALLOC_LIMIT = 8 /* topk_decode_noalloc: more rows than its fixed scratch holds */
} gvr_status;

/*
 * Decode top-K.  Row r belongs to request r / next_n and has
 *   n_r = (kv_lens[r / next_n] - next_n + r % next_n + 1) / compress_ratio
 * valid scores logits[r][0 .. n_r) (integer division), with n_r = 0 when
 * kv_lens[r / next_n] < next_n and n_r clamped to row_stride.  This is the MTP window formula
 * of "Block-skip fast path for self-sampling GVR top-K decode" (PR #18122, commit
 * "run_varlen"): kv_lens holds each request's total uncompressed cache length, and the
 * empty-row rule is from its commit "engine/reference convention alignment".
 *   kv_lens  int32 [ceil(num_rows / next_n)], device, read on the device only.
 *   indices  int32 [num_rows][k]: window indices (= column indices for decode), -1 pads; -2 in
 *            every slot of a row whose bounded wait gave up (see the conventions above).
 *   values   optional fp32 [num_rows][k]: the score at each returned index, bit-exact copied
 *            from logits; -FLT_MAX in -1 slots ("values output" commit of PR #18122).
 */
gvr_status topk_decode(const float* logits, int64_t row_stride, int64_t num_rows,
                       const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio, int32_t k,
                       int32_t* indices, float* values, void* stream);

/*
 * Prefill top-K.  Row r selects over the window [row_starts[r], row_ends[r]) of its own row
 * (compressed column units) and writes LOCAL indices (column - row_starts[r]) with a trailing
 * -1 pad; nv <= k yields the identity 0..nv-1 ("Self-sampling GVR V2 prefill indexer top-K",
 * PR #18702, section "Kernel").  The window start need not be 16-byte aligned: the loads start
 * at the aligned column below it and the lead lanes are excluded by position.  A start below 0
 * is treated as 0, an end beyond row_stride as row_stride, and an end at or before the start
 * as an empty window.
 *   row_starts, row_ends  int32 [num_rows], device.
 *   indices               int32 [num_rows][k]; -2 in every slot of a row whose bounded wait gave
 *                         up (see the conventions above).
 */
gvr_status topk_prefill(const float* logits, int64_t row_stride, int64_t num_rows,
                        const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                        int32_t* indices, void* stream);

/* Tuning and diagnostics for the *_ex entry points (the plain entry points use all zeros). */
enum {
  GVR_FLAG_FORCE_RESCUE = 1, /* skip the histogram: every long row takes the exact rescue */
  GVR_FLAG_NO_FLOOR = 2,     /* count every bin of the value histogram (no sampled floor) */
  GVR_FLAG_ZERO_CAP = 4,     /* candidate buffer of 0 slots: every long row overflows to rescue */
  GVR_FLAG_RADIX_REFINE = 8, /* refine every candidate set by radix select (not by ranking) */
  /* Deterministic mode ("Self-sampling GVR V2", the selection kernel's contract: exact
   * membership with smallest-index deterministic ties, optional output sorting): of the scores
   * equal to tau, the ones with the smallest window indices fill the remaining slots, so the
   * selected set is the same on every run.  Output order stays unspecified. */
  GVR_FLAG_DETERMINISTIC = 16,
  /* Deterministic ties, and each long row's k indices ordered by (score descending, window
   * index ascending), -0 equal to +0.  Rows with nv <= k keep the identity order 0..nv-1 and
   * the -1 pad. */
  GVR_FLAG_SORTED = 32,
  /* diagnostics: a crossing bin over the candidate buffer always takes the digit passes over
   * the row (no selection over per-CTA lists) */
  GVR_FLAG_STREAM_RESCUE = 64,
  /* the compact first-pass lists (1024 entries of score and 16-bit share position per CTA, 16
   * samples expected above tau) on every launch; by default the host picks them only where
   * they let a two-wave launch run as one wave with half the CTAs per row */
  GVR_FLAG_COMPACT_LISTS = 128,
  /* always the cluster kernel: for the *_ws entry points not the balanced kernel either (the
   * workspace is then not touched) */
  GVR_FLAG_CLUSTER_KERNEL = 256,
  /* diagnostics, *_ws entry points: the balanced kernel's last CTA of every long row selects the
   * row alone (the exact path it takes when the published scores cannot decide the row) */
  GVR_FLAG_SPLIT_ALONE = 512,
  /* *_ws entry points: the balanced kernel whenever the call fits it */
  GVR_FLAG_SPLIT_KERNEL = 1024,
  /* diagnostics: the first row's cluster reports a device-side give-up once its first pass is
   * complete (every bulk copy landed, no wait shortened) -- with GVR_FLAG_SHORT_KERNEL the
   * short-row kernel's CTA of row 0, once its window has landed -- so that row's indices become
   * -2 and its row_stats path GVR_PATH_DEVICE_ERROR while the other rows stay exact: the failure
   * path without a failure */
  GVR_FLAG_DIAG_FAIL_ROW0 = 2048,
  /* the short-row kernel for calls it takes (row_stride <= 16384, no flag but
   * GVR_FLAG_FORCE_RESCUE or GVR_FLAG_DIAG_FAIL_ROW0, no cluster or ring setting, not the hinted or block-skip entry
   * points; others run the cluster kernel) whatever the row count: one CTA of 1024 threads per
   * row stages the whole window in shared memory with bulk copies and selects over it.  Calls
   * with no flag take it by default when row_stride <= 16384 and the rows fit four waves of its
   * CTAs (two per SM), where it measured faster than the cluster kernel */
  GVR_FLAG_SHORT_KERNEL = 4096,
  /* topk_decode_blockskip: skip blocks whatever the samples estimate (the gate is not applied) */
  GVR_FLAG_BLOCKSKIP_ALWAYS = 8192
};

typedef struct gvr_options {
  int32_t cluster_size;       /* CTAs per row: 0 = automatic, else 1, 2, 4, 8 or 16 (16 is a
                                 non-portable cluster size: the launch fails where the device
                                 cannot schedule it; automatic use checks first) */
  int32_t ring_stages;        /* shared-memory ring stages of 4 KB per CTA: 0 = automatic,
                                 else 3..16 */
  int32_t flags;              /* GVR_FLAG_* bits; results stay exact under every flag */
  int32_t reserved;           /* must be 0 */
  int32_t* row_stats;         /* optional device int32 [num_rows][4]: path (GVR_PATH_*),
                                 candidate count m, histogram rounds (+10 when the row was
                                 read again to list the crossing bin), winners above the
                                 crossing bin */
} gvr_options;

/* Values of row_stats[r][0].  GVR_PATH_DEVICE_ERROR means a CTA gave up waiting (0.5 s) for
 * its staged scores; every index of that row is then -2.  It is not expected to happen. */
enum {
  GVR_PATH_DEVICE_ERROR = -1,
  GVR_PATH_SHORT = 0,           /* nv <= k: identity and -1 pad */
  GVR_PATH_REFINE = 1,          /* histogram, crossing bin, candidates, exact refine */
  GVR_PATH_RESCUE_BRACKET = 2,  /* invalid sampled bracket: exact rescue */
  GVR_PATH_RESCUE_OVERFLOW = 3, /* crossing bin exceeded the candidate buffer and some CTA's
                                   list overflowed: exact digit passes over the row, seeded
                                   with the crossing bin */
  GVR_PATH_RESCUE_FORCED = 4,   /* GVR_FLAG_FORCE_RESCUE */
  GVR_PATH_REFINE_CLUSTER = 5,  /* crossing bin exceeded the candidate buffer, every CTA's list
                                   held its counted scores: exact digit passes over the lists */
  GVR_PATH_REFINE_RELIST = 6,   /* crossing bin exceeded the candidate buffer and a first-pass
                                   list overflowed: one more read of the row lists the crossing
                                   bin and above per CTA, digit passes over those lists */
  GVR_PATH_SPLIT = 7,           /* balanced kernel: selected from the row's published scores */
  GVR_PATH_SPLIT_ALONE = 8,     /* balanced kernel: the row's last CTA selected it alone */
  GVR_PATH_NEG_INF_FILL = 9,    /* fewer than k scores above -inf: every other score is a winner,
                                   the remaining slots take -inf scores (tau = -inf), one pass */
  GVR_PATH_SHORT_KERNEL = 10,   /* short-row kernel: histogram, crossing bin, refine, all over the
                                   window staged in shared memory */
  GVR_PATH_SHORT_RADIX = 11     /* short-row kernel: exact radix select over the staged window
                                   (invalid bracket, floor too high, too many scores at or above
                                   it, crossing bin too big, forced rescue) */
};

/* topk_decode with tuning/diagnostic options (NULL = automatic, identical to topk_decode). */
gvr_status topk_decode_ex(const float* logits, int64_t row_stride, int64_t num_rows,
                          const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                          int32_t k, int32_t* indices, float* values, void* stream,
                          const gvr_options* options);

/* topk_prefill with tuning/diagnostic options (NULL = automatic, identical to topk_prefill). */
gvr_status topk_prefill_ex(const float* logits, int64_t row_stride, int64_t num_rows,
                           const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                           int32_t* indices, void* stream, const gvr_options* options);

/*
 * Decode top-K with hinted sampling (the request-level temporal hint of "Block-skip fast path
 * for self-sampling GVR top-K decode", PR #18122: the previous decode step's top-K indices of
 * each request, taken as-is, with no offset).  Identical results to topk_decode_ex: the hints
 * only choose the sampled positions that set the bracket and the first-pass floor.
 *   pre_idx         int32 [ceil(num_rows / next_n)][pre_idx_stride], device; row q holds the
 *                   window indices request q selected last step, shared by its next_n rows.
 *                   Entries outside [0, n_r) (the -1 pad, stale or garbage values) are
 *                   skipped; duplicates are allowed.  Only the first k entries of a row are read.
 *   pre_idx_stride  >= k (GVR_ERR_ARG otherwise); pre_idx 4-byte aligned (GVR_ERR_ALIGN),
 *                   non-NULL when num_rows > 0 (GVR_ERR_NULL).
 * Every other argument, the ownership rules and the errors are those of topk_decode_ex.
 */
gvr_status topk_decode_hinted(const float* logits, int64_t row_stride, int64_t num_rows,
                              const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                              int32_t k, const int32_t* pre_idx, int64_t pre_idx_stride,
                              int32_t* indices, float* values, void* stream,
                              const gvr_options* options);

/*
 * Decode top-K with a block-maxima side tensor (the opt-in block-skip row pass of "Block-skip
 * fast path for self-sampling GVR top-K decode", PR #18122, description and last commit): the
 * first counting pass reads only the 32-score blocks whose bound reaches the sampled floor.
 * Results are identical to topk_decode_ex for any valid bounds.
 *   block_max         fp32 [num_rows][block_max_stride], device: block_max[r][b] must be >= every
 *                     score of row r in columns [32 b, 32 b + 32) inside the row's window
 *                     [0, n_r) (the block's maximum is the usual producer output; a larger bound
 *                     only costs reads; NaN means "read the block").  Only blocks that meet the
 *                     window are read.
 *   block_max_stride  >= ceil(row_stride / 32) (GVR_ERR_ARG otherwise); block_max 4-byte
 *                     aligned (GVR_ERR_ALIGN), non-NULL when num_rows > 0 (GVR_ERR_NULL).
 * Gate (on the device, per row): once the sampled floor is known, the block64 samples give the
 * share of 32-score sample halves that reach it, an estimate of the share of blocks the skipping
 * pass would still read.  Above a quarter the row takes the ordinary staged pass (every block
 * read at the streaming rate, as topk_decode_ex); at or below it, the first ring stages of each
 * CTA's share (staged for every row at the start) are read whole and the rest block by block.
 * GVR_FLAG_BLOCKSKIP_ALWAYS skips the gate.  The later passes that need every score (the rare
 * second pass below the floor, the row-wide selection) read whole shares as usual.  Every other
 * argument, the ownership rules and the errors are those of topk_decode_ex.
 */
gvr_status topk_decode_blockskip(const float* logits, int64_t row_stride, int64_t num_rows,
                                 const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                                 int32_t k, const float* block_max, int64_t block_max_stride,
                                 int32_t* indices, float* values, void* stream,
                                 const gvr_options* options);

/*
 * Balanced entry points with a workspace.  A decode batch's rows can differ widely in length
 * (n_r from kv_lens, known only on the device), and the cluster kernel above sizes every row's
 * cluster from row_stride, so its longest rows set the time.  These entry points may instead
 * run the balanced kernel: every CTA reads all rows' lengths on the device, the batch's valid
 * scores are cut into chunks of one size, one CTA per chunk, and each chunk publishes the scores
 * at or above its row's sampled floor to the workspace; the last chunk of a row to finish
 * selects the row from them (histogram over the sampled bracket, crossing bin, exact refine), or
 * -- when they cannot decide it (fewer than k reached the floor, a chunk's slot overflowed, an
 * invalid bracket) -- selects the row alone by an exact radix select over the whole window.
 * Same method ("GVR K=2048 reg_clus with block64 sampling and parallel rescue", PR #20998,
 * "What changes"), same results: exact, tie-interchangeable, identical conventions.
 *
 * The balanced kernel runs when options->flags asks for it (GVR_FLAG_SPLIT_KERNEL or
 * GVR_FLAG_SPLIT_ALONE, and no other flag), num_rows <= 512 and num_rows is at most half its
 * grid (the device's SM count x 8 CTAs); otherwise the call is exactly topk_decode_ex /
 * topk_prefill_ex and the workspace is not touched (GVR_FLAG_CLUSTER_KERNEL forces that).
 *
 * The workspace is device memory the caller owns, at least gvr_workspace_size bytes, 16-byte
 * aligned, and ZERO-FILLED before its first use (cudaMemset once); every call that completes
 * leaves it zero-filled again.  Calls that can overlap on the GPU (different streams without an
 * ordering between them) must use different workspaces.  Every other argument, the ownership
 * rules and the errors are those of topk_decode_ex / topk_prefill_ex, plus GVR_ERR_WORKSPACE.
 */
/* Bytes of workspace the *_ws entry points need on the current device (sm_count <= 0) or on a
 * GB300-class device with sm_count SMs; the size does not depend on the call's shape. */
gvr_status gvr_workspace_size(int32_t sm_count, size_t* bytes);

gvr_status topk_decode_ws(const float* logits, int64_t row_stride, int64_t num_rows,
                          const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                          int32_t k, int32_t* indices, float* values, void* workspace,
                          size_t workspace_bytes, void* stream, const gvr_options* options);

gvr_status topk_prefill_ws(const float* logits, int64_t row_stride, int64_t num_rows,
                           const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                           int32_t* indices, void* workspace, size_t workspace_bytes, void* stream,
                           const gvr_options* options);

/*
 * Decode top-K that allocates nothing and needs no workspace from the caller.  This entry point
 * has no counterpart in the pages; it exists for callers that cannot allocate device memory
 * when they select: an inference engine's plugin or op that is only handed its inputs and
 * outputs at enqueue time and must not call cudaMalloc there, a serving loop on a fixed memory
 * arena owned by another allocator, or latency-critical code that cannot afford the device-wide
 * synchronization cudaMalloc may cause.
 *
 * It runs the balanced kernel of topk_decode_ws (same method, same exact results, same argument
 * rules and errors as topk_decode) on a scratch area the library itself holds: a fixed device
 * array of about 8 MB, present on every device that loads the library until the process exits.
 * Limits and behaviour:
 *   - num_rows must be at most GVR_NOALLOC_MAX_ROWS (128); more returns GVR_ERR_NOALLOC_LIMIT
 *     before anything is enqueued.
 *   - The first call on a device looks up the array's device address (once per device, with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array.  Each call clears its row counters on `stream` first (one
 *     small memset, then the kernel), but calls that overlap on the GPU -- different streams
 *     without an ordering between them, or different host threads -- race on the array and may
 *     return wrong results; order them, or use topk_decode_ws with one workspace each.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine is called.
 */
#define GVR_NOALLOC_MAX_ROWS 128
gvr_status topk_decode_noalloc(const float* logits, int64_t row_stride, int64_t num_rows,
                               const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                               int32_t k, int32_t* indices, float* values, void* stream);

/* Static English text for a status code; never NULL. */
const char* gvr_status_string(gvr_status status);

/*
 * The launch geometry the library would choose for a plain topk_decode / topk_prefill call on
 * the current device (host only, no device work): CTAs per row (cluster size), 4 KB stages of
 * each CTA's shared-memory ring, threads per CTA and dynamic shared memory bytes per CTA.  The
 * short-row kernel (see GVR_FLAG_SHORT_KERNEL) reads as cluster size 1, ring stages 0 and
 * 1024 threads.  Returns the GVR_ERR_* code
 * the entry points would return for these arguments.  sm_count > 0 plans for a GB300-class
 * device with that many SMs (228 KB shared memory per SM) without touching a device; any
 * output pointer may be NULL.
 */
gvr_status gvr_plan(int64_t row_stride, int64_t num_rows, int32_t k, const gvr_options* options,
                    int32_t sm_count, int32_t* cluster_size, int32_t* ring_stages, int32_t* threads,
                    int32_t* smem_bytes);

#ifdef __cplusplus
}
#endif

#endif /* GVR_TOPK_H */
