/*
 * gvr_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, obviously correct CPU oracle for the exact per-row top-K that
 * the DSA sparse-attention indexer selects.  Only tests/, the smoke check in
 * __graft_entry__ and the cpu_baseline / reference leg of bench.py may load
 * this library.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the plain definition the GVR method reaches exactly):
 *   "Self-sampling GVR V2 prefill indexer top-K" (TensorRT-LLM PR #18702),
 *   section "Kernel": per row r the top-K of logits[r, ks:ke], written in the
 *   local frame (column - ks) with a trailing -1 pad, identity 0..nv-1 when
 *   nv = ke - ks <= k.
 *   "Block-skip fast path for self-sampling GVR top-K decode" (PR #18122),
 *   commit "run_varlen": decode rows take n = (kv_len - next_n + row % next_n
 *   + 1) / compress_ratio valid scores, kv_lens is per request (row / next_n);
 *   commit "engine/reference convention alignment": kv_len < next_n is an
 *   empty row (all -1); commit "values output": optional fp32 values, short
 *   rows copy the head and pad with -FLT_MAX; the contract is "exact
 *   (tie-interchangeable) top-K" with signed zeros normalized; NaN inside
 *   the window is outside the contract (this oracle refuses such rows).
 *
 * Method of this oracle: copy the window, normalize -0 to +0, sort all
 * (value, window index) pairs by value descending then index ascending with
 * the C library qsort, keep the first K.  Ties at the K-th value tau are
 * therefore broken by the smallest window index; any other choice among the
 * tied entries is equally correct, and the tests compare tie-aware.
 *
 * Parity is pinned (tests/test_oracle_pins.py) by brute force over all
 * K-subsets of tiny rows, the invariant count(>tau) < K <= count(>=tau),
 * numpy's partition on random rows, closed forms (all-equal, two-valued,
 * -inf/+inf classes, signed zero, short-row identity, the decode length
 * formula on hand-computed points) and a translation invariance for the
 * prefill lead.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NAN_IN_WINDOW = 2, ORACLE_NO_MEMORY = 3 };

typedef struct {
  float v;   /* score with -0 normalized to +0 */
  int32_t j; /* window-local index */
} oracle_pair;

/* Order: larger value first; among equal values, smaller index first. */
static int oracle_pair_order(const void *pa, const void *pb) {
  const oracle_pair *a = (const oracle_pair *)pa;
  const oracle_pair *b = (const oracle_pair *)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  if (a->j < b->j) return -1;
  if (a->j > b->j) return 1;
  return 0;
}

/*
 * Decode row length, "run_varlen" commit of PR #18122: the request of row r
 * is r / next_n; its n = (kv_len - next_n + r % next_n + 1) / compress_ratio
 * (C division of a positive numerator); a request with kv_len < next_n has
 * empty rows.  n is clamped to the row stride (the "envelope clamp" of the
 * register-family commit).
 */
int64_t oracle_decode_row_len(int64_t r, const int32_t *kv_lens, int32_t next_n,
                              int32_t compress_ratio, int64_t row_stride) {
  int64_t kv = kv_lens[r / next_n];
  if (kv < next_n) return 0;
  int64_t num = kv - next_n + (r % next_n) + 1;
  int64_t n = num / compress_ratio;
  if (n > row_stride) n = row_stride;
  return n;
}

/*
 * Prefill window, "Kernel" section of PR #18702: [ks, ke) in compressed
 * column units.  Starts below 0 and ends past the stride are clamped to the
 * row; an end before the start is an empty window.
 */
static void oracle_prefill_window(int64_t ks, int64_t ke, int64_t row_stride, int64_t *a,
                                  int64_t *nv) {
  if (ks < 0) ks = 0;
  if (ke > row_stride) ke = row_stride;
  *a = ks;
  *nv = ke > ks ? ke - ks : 0;
}

/*
 * Exact top-K of one window w[0..nv).  Writes k indices (and optionally the
 * k values gathered from the window) and tau, the K-th largest value after
 * signed-zero normalization (NaN when nv <= k, where no selection happens).
 * scratch must hold nv pairs.
 */
static int oracle_select_window(const float *w, int64_t nv, int32_t k, int32_t *out, float *vals,
                                float *tau, oracle_pair *scratch) {
  if (nv <= k) {
    for (int64_t i = 0; i < k; ++i) {
      out[i] = i < nv ? (int32_t)i : -1;
      if (vals) vals[i] = i < nv ? w[i] : -FLT_MAX;
    }
    if (tau) *tau = NAN;
    return ORACLE_OK;
  }
  for (int64_t j = 0; j < nv; ++j) {
    float v = w[j];
    if (isnan(v)) return ORACLE_NAN_IN_WINDOW;
    scratch[j].v = (v == 0.0f) ? 0.0f : v;
    scratch[j].j = (int32_t)j;
  }
  qsort(scratch, (size_t)nv, sizeof(oracle_pair), oracle_pair_order);
  for (int32_t i = 0; i < k; ++i) {
    out[i] = scratch[i].j;
    if (vals) vals[i] = w[scratch[i].j];
  }
  if (tau) *tau = scratch[k - 1].v;
  return ORACLE_OK;
}

static int oracle_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* Number of threads the row loop would use for a request of nthreads. */
int oracle_thread_count(int nthreads) { return oracle_threads(nthreads); }

/*
 * Decode top-K over rows [0, num_rows).  logits is [num_rows, row_stride]
 * fp32, kv_lens has ceil(num_rows / next_n) entries, indices is
 * [num_rows, k], values (nullable) is [num_rows, k], tau (nullable) is
 * [num_rows].  nan_row (nullable) receives the first row refused for a NaN
 * inside its window.
 */
int oracle_topk_decode(const float *logits, int64_t row_stride, int64_t num_rows,
                       const int32_t *kv_lens, int32_t next_n, int32_t compress_ratio,
                       int32_t k, int32_t *indices, float *values, float *tau,
                       int nthreads, int64_t *nan_row) {
  if (!logits || !kv_lens || !indices || row_stride < 1 || num_rows < 0 || next_n < 1 ||
      compress_ratio < 1 || k < 1)
    return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  int64_t first_bad = -1;
  int nt = oracle_threads(nthreads);
  (void)nt;
#pragma omp parallel num_threads(nt)
  {
    oracle_pair *scratch = (oracle_pair *)malloc(sizeof(oracle_pair) * (size_t)row_stride);
    if (!scratch) {
#pragma omp critical
      status = ORACLE_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < num_rows; ++r) {
      if (!scratch) continue;
      int64_t n = oracle_decode_row_len(r, kv_lens, next_n, compress_ratio, row_stride);
      int rc = oracle_select_window(logits + r * row_stride, n, k, indices + r * k,
                                    values ? values + r * k : NULL, tau ? tau + r : NULL, scratch);
      if (rc != ORACLE_OK) {
#pragma omp critical
        {
          if (status == ORACLE_OK || status == ORACLE_NAN_IN_WINDOW) {
            status = rc;
            if (first_bad < 0 || r < first_bad) first_bad = r;
          }
        }
      }
    }
    free(scratch);
  }
  if (nan_row) *nan_row = first_bad;
  return status;
}

/*
 * Prefill top-K over rows [0, num_rows): row r selects over
 * logits[r, row_starts[r] : row_ends[r]] and writes window-local indices.
 */
int oracle_topk_prefill(const float *logits, int64_t row_stride, int64_t num_rows,
                        const int32_t *row_starts, const int32_t *row_ends, int32_t k,
                        int32_t *indices, float *tau, int nthreads, int64_t *nan_row) {
  if (!logits || !row_starts || !row_ends || !indices || row_stride < 1 || num_rows < 0 || k < 1)
    return ORACLE_BAD_ARG;
  int status = ORACLE_OK;
  int64_t first_bad = -1;
  int nt = oracle_threads(nthreads);
  (void)nt;
#pragma omp parallel num_threads(nt)
  {
    oracle_pair *scratch = (oracle_pair *)malloc(sizeof(oracle_pair) * (size_t)row_stride);
    if (!scratch) {
#pragma omp critical
      status = ORACLE_NO_MEMORY;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < num_rows; ++r) {
      if (!scratch) continue;
      int64_t a, nv;
      oracle_prefill_window(row_starts[r], row_ends[r], row_stride, &a, &nv);
      int rc = oracle_select_window(logits + r * row_stride + a, nv, k, indices + r * k, NULL,
                                    tau ? tau + r : NULL, scratch);
      if (rc != ORACLE_OK) {
#pragma omp critical
        {
          if (status == ORACLE_OK || status == ORACLE_NAN_IN_WINDOW) {
            status = rc;
            if (first_bad < 0 || r < first_bad) first_bad = r;
          }
        }
      }
    }
    free(scratch);
  }
  if (nan_row) *nan_row = first_bad;
  return status;
}

/* Single window, any k >= 1: the selection core on its own, for the pins. */
int oracle_topk_window(const float *w, int64_t nv, int32_t k, int32_t *out, float *vals,
                       float *tau) {
  if ((!w && nv > 0) || !out || nv < 0 || k < 1) return ORACLE_BAD_ARG;
  oracle_pair *scratch = (oracle_pair *)malloc(sizeof(oracle_pair) * (size_t)(nv > 0 ? nv : 1));
  if (!scratch) return ORACLE_NO_MEMORY;
  int rc = oracle_select_window(w, nv, k, out, vals, tau, scratch);
  free(scratch);
  return rc;
}
