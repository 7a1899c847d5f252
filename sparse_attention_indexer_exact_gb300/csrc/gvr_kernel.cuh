// gvr_kernel.cuh -- the GVR (Guess-Verify-Refine) exact per-row top-K kernel for sm_103a.
//
// One thread-block cluster selects one row.  The row's valid window is split evenly over the
// cluster's CTAs; each CTA streams its share through a small ring of shared-memory stages
// filled by bulk asynchronous copies (TMA, completion on one mbarrier per stage), so the row
// is read from HBM once and each CTA needs little shared memory: several CTAs -- several rows
// -- are resident on every SM at a time.  Per row:
//
//   Guess   uniform block64 sampling: runs of 64 consecutive scores whose starts spread
//           evenly over the window, first run at 0, last run ending at nv -- K/64 runs, as in
//           "GVR K=2048 reg_clus with block64 sampling and parallel rescue" (TensorRT-LLM PR
//           #20998, "What changes"), or more when K is small against nv (at most 32).
//           GMIN / GMAX are the smallest / largest finite sample.
//   Verify  a value histogram of NB bins over [GMIN, GMAX] (values above GMAX saturate into
//           the top bin, below GMIN into bin 0; when a few far samples stretch the bins, they
//           end lower, at a robust sample rank); its cluster-wide suffix sums locate the bin
//           b* that crosses the K-th largest value tau ("Why the GLM row overflows").
//   Refine  scores in bins above b* are winners and are written at once; the m members of
//           b* go to a bounded candidate buffer in cluster rank 0, which picks the remaining
//           need = K - above winners exactly.  When m exceeds the buffer, the same exact
//           selection as the rescue runs over the CTAs' lists of counted scores instead of
//           the row (re-built by one more read when a list overflowed).
//   Rescue  an invalid bracket (no finite sample, or GMIN == GMAX) or a crossing bin that no
//           list can hold sends the row to an exact radix select over the 32-bit
//           order-preserving keys, 8-bit digit passes whose digit histograms are summed over
//           all CTAs of the cluster through distributed shared memory -- the parallel rescue of
//           PR #20998, in the same launch, with no host synchronization.  After a valid
//           histogram only the crossing bin's members take part.
//
// Implementation choices that keep the per-score work to about one compare:
//  * sampled histogram floor: the samples also give a floor t with a Poisson margin above the
//    expected K-th sample; only scores >= t are counted, and they are kept in per-warp
//    shared-memory lists for the collect step (no second read of the row).  Bins above bin(t)
//    are then complete, bin(t) itself is partial.  Only when fewer than K scores reach t are
//    the scores below it counted in a second pass, so the result never depends on the floor.
//  * no warp collective per stage in the first pass: a thread with hits takes list slots with
//    one shared atomic on its warp's counter; the hits' bins are counted after the pass, from
//    the list (hits past a full list in a per-thread register run of one bin).  A tie class
//    above the floor -- every counted score one value -- is recognised from the cluster's
//    smallest and largest counted key, and its slots come from the lists.
//  * the first pass's histogram reaches every CTA of the cluster as TMA bulk reductions into
//    shared memory, counted on an mbarrier (no cluster barrier).
//  * six instantiations: the plain one, the extended modes (deterministic ties by smallest
//    index and sorted output, hinted sampling, the block-skip first pass) or the block-skip
//    first pass alone; each with or without the compact lists (L16: 1024 entries of score and
//    16-bit share position instead of 768 of score and index, chosen by the host where they
//    let half as many CTAs hold a row's list).
//
// The bin function is monotone non-decreasing in the score (IEEE round-to-nearest subtract and
// multiply by a positive scale, clamp, truncate), which is all the crossing-bin logic needs;
// it is evaluated with the same instruction sequence everywhere, so every pass and every CTA
// classifies a score identically.  Positions outside the window (the lead lanes below an
// unaligned window start, the lanes past its end) are excluded by position in every pass.
#pragma once

#include <cfloat>
#include <cstddef>
#include <cstdint>

#include "gvr_device.cuh"

namespace gvr {

constexpr int THREADS = 128;          // threads per CTA
constexpr int NB = 1024;              // value-histogram bins over [GMIN, GMAX]
constexpr int VPS = 2;                // float4 per thread per stage
constexpr int STAGE_VEC = THREADS * VPS;  // 256 float4 = 4 KB per stage
constexpr int MIN_STAGES = 3;         // ring depth bounds (the host picks the depth per launch)
constexpr int MAX_STAGES = 16;
constexpr int LIST_BYTES = 6144;      // the per-CTA list of above-floor scores kept for the collect
// Two list formats in the same bytes: (score, 32-bit window index) -- 768 entries -- or
// (score, 16-bit position in the CTA's share) -- 1024 entries, for shares of at most
// LIST_MAX_STAGES stages (the compact format, chosen by the host for long shares).
constexpr int LIST_CAP = LIST_BYTES / 8;
constexpr int LIST_CAP16 = LIST_BYTES / 6;
constexpr int LIST_MAX_STAGES = 64;
constexpr int CAP = 512;              // candidate slots in cluster rank 0
constexpr uint32_t REC_CAP = LIST_BYTES / 4;  // window indices the first rescue digit pass records
constexpr int RING_CAND = STAGE_VEC * 16 / 8;  // (score, index) candidates one idle ring stage holds
constexpr int BULK_BINS = 512;       // first-pass counts of at most this many bins go as bulk adds
constexpr int RANK_REFINE_MAX = 256;
constexpr uint32_t UNLISTED_RANK0 = 1u << 16;  // marks rank 0's overflowed list in the count  // m at or below: refine by pairwise ranking
constexpr int MAX_K = 2048;
constexpr int MAX_SAMPLES = 2048;     // block64 samples per row at most (32 runs, one per lane)

// Samples of a long row (nv > k): k (the k / 64 runs of uniform block64 sampling), or more
// when k is small against nv -- enough runs, up to MAX_SAMPLES, that about mu_target (8, or 16
// for the compact lists' long shares) samples are expected above the K-th score.  The floor keeps a margin of a few
// samples over that expectation, so with fewer samples it would count and list several times
// K scores.
__host__ __device__ constexpr uint32_t sample_count(uint32_t k, uint32_t nv, uint32_t mu_target = 8) {
  const uint32_t per = 64u * k / mu_target;              // row scores per run for that target
  const uint32_t runs = (nv + per - 1u) / per;           // nv < 2^31, per <= 16384
  const uint32_t n = 64u * runs;
  return n <= k ? k : (n >= uint32_t(MAX_SAMPLES) ? uint32_t(MAX_SAMPLES) : n);
}

constexpr uint64_t WAIT_LIMIT_NS = 500000000ull;  // bound on any wait for staged data (0.5 s)

enum : int32_t { MODE_DECODE = 0, MODE_PREFILL = 1 };
enum : int32_t {
  FLAG_FORCE_RESCUE = 1,
  FLAG_NO_FLOOR = 2,
  FLAG_ZERO_CAP = 4,
  FLAG_RADIX_REFINE = 8,
  FLAG_DETERMINISTIC = 16,
  FLAG_SORTED = 32,
  FLAG_STREAM_RESCUE = 64,
  FLAG_COMPACT_LISTS = 128,
  FLAG_DIAG_FAIL_ROW0 = 2048,
  FLAG_BLOCKSKIP_ALWAYS = 8192
};
enum : int32_t {
  PATH_DEVICE_ERROR = -1,
  PATH_SHORT = 0,
  PATH_REFINE = 1,
  PATH_RESCUE_BRACKET = 2,
  PATH_RESCUE_OVERFLOW = 3,
  PATH_RESCUE_FORCED = 4,
  PATH_REFINE_CLUSTER = 5,
  PATH_REFINE_RELIST = 6,
  PATH_NEG_INF_FILL = 9
};

struct Params {
  const float* logits;
  int64_t row_stride;
  const int32_t* kv_lens;     // decode
  const int32_t* row_starts;  // prefill
  const int32_t* row_ends;    // prefill
  const int32_t* pre_idx;     // decode, optional: sample positions per request
  int64_t pre_stride;         // row stride of pre_idx (>= k)
  const float* block_max;     // decode, optional: an upper bound of every 32-score block
  int64_t bmax_stride;        // row stride of block_max (>= ceil(row_stride / 32))
  int32_t* indices;
  float* values;              // nullable
  int32_t* row_stats;         // nullable, [rows][4]
  int32_t next_n;
  int32_t compress_ratio;
  int32_t k;
  int32_t mode;
  int32_t flags;
  int32_t nstage;             // ring depth, MIN_STAGES..MAX_STAGES
};

struct Crossing {
  int32_t bin;          // b*
  uint32_t above;       // cluster-wide count in bins above b*
  uint32_t m;           // cluster-wide count in b*
  uint32_t my_above;    // this CTA's count in bins above b*
  uint32_t my_cand;     // this CTA's count in b*
  uint32_t total;       // cluster-wide count over all bins
};

struct alignas(16) Smem {
  uint32_t wsum[2][8];
  float wmin[8];
  float whmin[8], whmax[8];        // hinted sampling: smallest / largest finite hinted score per warp
  uint32_t whcnt[8];               // hinted sampling: in-window hints per warp
  float hpart_min, hpart_max;      // this CTA's share of the hints (read by the whole cluster)
  uint32_t hpart_cnt;
  float hagg_min, hagg_max;        // the cluster's hints
  uint32_t hagg_cnt;
  float wmax[8];
  float4 tail;                     // the partial last vector of the window, NaN-padded
  Crossing cross;
  float vthr, vthr1;
  int32_t fpart;
  uint32_t dsel, dabove, dcnt, dmy_above, dmy_at;
  uint32_t kmin_loc, kmax_loc;     // rescue: smallest / largest key of this CTA's matching scores
  uint32_t list_n[THREADS / 32];   // scores each warp appended to its segment (may exceed it)
  uint32_t unlisted;               // CTAs of the cluster whose list overflowed (each adds 1; rank 0
                                   // adds 1 + UNLISTED_RANK0)
  uint32_t relist_n;               // scores of the crossing bin and above listed again
  uint32_t relist_bad;             // CTAs of the cluster whose second list overflowed
  uint32_t klo, khi;               // order keys bounding the crossing bin's members
  uint32_t ctr_win, ctr_cand;      // this CTA's slot counters (refine path)
  uint32_t gctr_above, gctr_cand;  // rank 0: hands out each CTA's winner / candidate slot bases
  uint32_t base_above, base_cand;  // this CTA's slot bases
  uint32_t ctr_rwin, ctr_rtie;     // rank 0's counters for its own radix refine
  uint32_t rc_win, rc_tie;         // rank 0's counters shared by the cluster in rescue
  uint32_t saved;                  // count of the partial floor bin before the second pass
  uint32_t rec_n;                  // rescue: members recorded in the first digit pass (may exceed REC_CAP)
  uint32_t hk_min, hk_max;         // the cluster's smallest / largest order key of the first pass's
                                   // scores >= thr (every CTA adds its own)
  uint32_t hlisted;                // the cluster's listed first-pass scores
  uint32_t end_hits, nbr_hits;     // samples at or above the floor's bin in the end runs / their neighbours
  uint32_t tout;                   // this CTA gave up waiting for staged data
  uint32_t err;                    // rank 0: some CTA of the cluster gave up
  uint64_t bar[MAX_STAGES];        // one mbarrier per ring stage
  uint64_t hbar;                   // completes once every CTA's first-pass counts have landed in tot
  // Last members: hist, tot and the list, then (after padding) the ring -- one contiguous area
  // that rank 0 reuses at the very end for the sort keys of the sorted output.
  alignas(16) uint32_t hist[NB + 4];  // this CTA's counts (groups of 4 bins read as 16-byte
                                      // vectors); hist[NB]: 1 when this CTA's list overflowed
  uint32_t tot[NB + 4];            // cluster-wide counts, added here by every CTA of the cluster
                                   // (tot[NB]: CTAs whose list overflowed); the rescue's two
                                   // 256-bin digit histograms reuse it
  union {  // the first-pass list, in one of its two formats
    struct {
      float list_v[LIST_CAP];
      int32_t list_j[LIST_CAP];
    };
    struct {
      float list_v16[LIST_CAP16];
      uint16_t list_p16[LIST_CAP16];  // stage of the share * 1024 + offset in the stage
    };
  };
};
static_assert(offsetof(Smem, hist) % 16 == 0 && offsetof(Smem, tot) % 16 == 0,
              "histograms are read as 16-byte vectors");
static_assert(offsetof(Smem, bar) % 8 == 0, "mbarriers must be 8-byte aligned");
static_assert(2 * 256 + 4 <= NB, "the rescue's digit totals and key bounds live in tot");
static_assert(RING_CAND >= CAP, "one ring stage holds the candidate buffer");
static_assert(sizeof(float) * LIST_CAP + sizeof(int32_t) * LIST_CAP == 4 * REC_CAP,
              "the rescue's record fills exactly the list area");

__device__ __forceinline__ uint32_t* digit_hist(Smem& S, int buf) { return S.tot + 256 * buf; }

template <int N>
struct IntC {
  static constexpr int value = N;
};

// Dynamic shared memory: the fixed part, then the ring of nstage stages (bulk-copy
// destinations, 128-byte aligned).
constexpr int SMEM_FIXED = int((sizeof(Smem) + 127) / 128 * 128);
__host__ __device__ constexpr int smem_bytes(int nstage) { return SMEM_FIXED + nstage * STAGE_VEC * 16; }
static_assert(int(offsetof(Smem, hist)) + int(sizeof(uint64_t)) * MAX_K <= smem_bytes(MIN_STAGES),
              "the sort keys fit from hist to the end of the smallest ring");

// Monotone bin of a score in [GMIN, GMAX] with NB bins; NaN maps to bin 0.
__device__ __forceinline__ int value_bin(float v, float gmin, float sc) {
  float x = __fmul_rn(__fsub_rn(v, gmin), sc);
  x = fminf(fmaxf(x, 0.0f), float(NB - 1));
  return __float2int_rz(x);
}

// Smallest float v (non-NaN) with value_bin(v) >= fbin, for 1 <= fbin <= NB-1.  Warp-collective:
// all 32 lanes must call it.  Each round probes 32 evenly spaced keys of the current interval,
// so the interval shrinks 32x per round (7 rounds cover the 2^32 key space).
__device__ __forceinline__ float floor_value(int fbin, float gmin, float sc) {
  const int lane = threadIdx.x & 31;
  uint32_t lo = KEY_NEG_INF;  // bin(-inf) = 0 < fbin
  uint32_t hi = KEY_POS_INF;  // bin(+inf) = NB-1 >= fbin
  for (int round = 0; round < 40 && hi - lo > 1; ++round) {
    const uint64_t span = uint64_t(hi - lo);
    const uint32_t probe = lo + uint32_t((span * uint64_t(lane + 1)) >> 5);  // lane 31 probes hi
    const bool t = value_bin(key_to_float(probe), gmin, sc) >= fbin;
    const unsigned m = __ballot_sync(FULL_MASK, t);  // monotone: a suffix of the lanes
    const int first = __ffs(m) - 1;
    const uint32_t nhi = __shfl_sync(FULL_MASK, probe, first);
    const uint32_t plo = __shfl_sync(FULL_MASK, probe, first > 0 ? first - 1 : 0);
    lo = first > 0 ? plo : lo;
    hi = nhi;
  }
  return key_to_float(hi);
}

// Warp-aggregated slot allocation: lanes with `want` set get consecutive values of *ctr
// (shared memory of this CTA).  Warp-collective.
__device__ __forceinline__ uint32_t warp_alloc_local(uint32_t* ctr, bool want) {
  const unsigned mask = __ballot_sync(FULL_MASK, want);
  uint32_t base = 0;
  if (mask) {
    const int leader = __ffs(mask) - 1;
    if ((threadIdx.x & 31) == leader) base = atomicAdd(ctr, uint32_t(__popc(mask)));
    base = __shfl_sync(FULL_MASK, base, leader);
  }
  return base + __popc(mask & lanemask_lt());
}

// Warp-aggregated allocation of n < 16 consecutive slots per lane from *ctr (shared memory of
// this CTA): returns the lane's first slot.  Warp-collective.
__device__ __forceinline__ uint32_t warp_alloc_n(uint32_t* ctr, uint32_t n) {
  const unsigned lt = lanemask_lt();
  uint32_t excl = 0, tot = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const unsigned m = __ballot_sync(FULL_MASK, (n >> b) & 1u);
    excl += uint32_t(__popc(m & lt)) << b;
    tot += uint32_t(__popc(m)) << b;
  }
  uint32_t base = 0;
  if (tot) {  // warp-uniform
    if ((threadIdx.x & 31) == 0) base = atomicAdd(ctr, tot);
    base = __shfl_sync(FULL_MASK, base, 0);
  }
  return base + excl;
}

// Find the crossing bin in the cluster-wide totals S.tot: the highest b with
// sum_{bins >= b} tot >= k, with this CTA's own counts above and at b (from S.hist).  Thread t
// owns the NB/T bins NB-1-(NB/T)t down to NB-(NB/T)(t+1), so thread order is descending order.
template <int T, class SM>
__device__ __forceinline__ Crossing scan_crossing(SM& S, uint32_t k) {
  constexpr int BPT = NB / T;
  constexpr int NW = T / 32;
  static_assert(BPT % 4 == 0 && NW <= 8, "bins per thread must be a multiple of 4");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo_bin = NB - BPT * (tid + 1);
  uint32_t tot[BPT], loc[BPT];
#pragma unroll
  for (int q = 0; q < BPT / 4; ++q) {
    const uint4 t4 = *reinterpret_cast<const uint4*>(&S.tot[lo_bin + 4 * q]);
    const uint4 l4 = *reinterpret_cast<const uint4*>(&S.hist[lo_bin + 4 * q]);
    const uint32_t tw[4] = {t4.x, t4.y, t4.z, t4.w};
    const uint32_t lw[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tot[BPT - 1 - (4 * q + e)] = tw[e];  // descending position of bin lo_bin + 4q + e
      loc[BPT - 1 - (4 * q + e)] = lw[e];
    }
  }
  uint32_t st = 0, sl = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    st += tot[j];
    sl += loc[j];
  }
  uint32_t it = st, il = sl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(FULL_MASK, it, o);
    const uint32_t b = __shfl_up_sync(FULL_MASK, il, o);
    if (lane >= o) {
      it += a;
      il += b;
    }
  }
  if (lane == 31) {
    S.wsum[0][warp] = it;
    S.wsum[1][warp] = il;
  }
  __syncthreads();
  uint32_t wt = 0, wl = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t x = S.wsum[0][w];
    if (w < warp) {
      wt += x;
      wl += S.wsum[1][w];
    }
    total += x;
  }
  const uint32_t et = wt + it - st;  // cluster-wide count in bins above this thread's bins
  const uint32_t el = wl + il - sl;  // this CTA's count there
  if (et < k && et + st >= k) {
    uint32_t cum = et, cl = el;
    bool found = false;  // predicated, not break: the loop stays unrolled, the arrays in registers
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      if (!found && cum + tot[j] >= k) {
        S.cross.bin = lo_bin + BPT - 1 - j;
        S.cross.above = cum;
        S.cross.m = tot[j];
        S.cross.my_above = cl;
        S.cross.my_cand = loc[j];
        found = true;
      }
      cum += tot[j];
      cl += loc[j];
    }
  }
  __syncthreads();
  Crossing r = S.cross;
  r.total = total;
  return r;
}

// The highest bin b of arr[0..NB) with sum_{bins >= b} arr >= want, or -1 when the total is
// below want.  Block-collective; thread t owns bins NB-1-(NB/T)t down to NB-(NB/T)(t+1).
template <int T, class SM>
__device__ __forceinline__ int suffix_cross(SM& S, const uint32_t* arr, uint32_t want) {
  constexpr int BPT = NB / T;
  constexpr int NW = T / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo_bin = NB - BPT * (tid + 1);
  static_assert(BPT % 4 == 0, "bins per thread are read as 16-byte vectors (arr 16-byte aligned)");
  uint32_t c[BPT];
  uint32_t st = 0;
#pragma unroll
  for (int q = 0; q < BPT / 4; ++q) {
    const uint4 v = *reinterpret_cast<const uint4*>(arr + lo_bin + 4 * q);
    c[BPT - 1 - 4 * q] = v.x;  // descending position of bin lo_bin + 4q + e
    c[BPT - 2 - 4 * q] = v.y;
    c[BPT - 3 - 4 * q] = v.z;
    c[BPT - 4 - 4 * q] = v.w;
    st += v.x + v.y + v.z + v.w;
  }
  uint32_t it = st;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(FULL_MASK, it, o);
    if (lane >= o) it += a;
  }
  if (lane == 31) S.wsum[0][warp] = it;
  if (tid == 0) S.dsel = 0xffffffffu;
  __syncthreads();
  uint32_t before = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w)
    if (w < warp) before += S.wsum[0][w];
  const uint32_t ex = before + it - st;
  if (ex < want && ex + st >= want) {
    uint32_t cum = ex;
    bool found = false;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      cum += c[j];
      if (!found && cum >= want) {
        S.dsel = uint32_t(lo_bin + BPT - 1 - j);
        found = true;
      }
    }
  }
  __syncthreads();
  const int r = int(S.dsel);
  __syncthreads();
  return r;
}

struct DigitCross {
  uint32_t digit;     // d*
  uint32_t above;     // cluster-wide count of digits above d* (among the matching keys)
  uint32_t cnt;       // cluster-wide count at d*
  uint32_t my_above;  // this CTA's count above d*
  uint32_t my_at;     // this CTA's count at d*
  uint32_t my_all;    // this CTA's count over every digit (its matching keys)
};

// Digit crossing over pushed cluster-wide digit counts dtot (local) and this CTA's own counts
// dloc: the digit d (scanning from 255 down) where the running cluster count reaches `need`.
// Thread t owns digits 255 - DPT t down to 256 - DPT (t + 1).
template <int T, class SM>
__device__ __forceinline__ DigitCross digit_scan(SM& S, const uint32_t* dtot, const uint32_t* dloc,
                                                 uint32_t need) {
  constexpr int DPT = 256 / T;
  constexpr int NW = T / 32;
  static_assert(DPT * T == 256 && NW <= 8, "threads must divide 256");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t tot[DPT], loc[DPT];
  uint32_t st = 0, sl = 0;
#pragma unroll
  for (int j = 0; j < DPT; ++j) {
    const int d = 255 - DPT * tid - j;
    tot[j] = dtot[d];
    loc[j] = dloc[d];
    st += tot[j];
    sl += loc[j];
  }
  uint32_t it = st, il = sl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(FULL_MASK, it, o);
    const uint32_t b = __shfl_up_sync(FULL_MASK, il, o);
    if (lane >= o) {
      it += a;
      il += b;
    }
  }
  if (lane == 31) {
    S.wsum[0][warp] = it;
    S.wsum[1][warp] = il;
  }
  __syncthreads();
  uint32_t wt = 0, wl = 0, all = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    if (w < warp) {
      wt += S.wsum[0][w];
      wl += S.wsum[1][w];
    }
    all += S.wsum[1][w];
  }
  const uint32_t et = wt + it - st, el = wl + il - sl;
  if (et < need && et + st >= need) {
    uint32_t cum = et, cl = el;
    bool found = false;
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      if (!found && cum + tot[j] >= need) {
        S.dsel = uint32_t(255 - DPT * tid - j);
        S.dabove = cum;
        S.dcnt = tot[j];
        S.dmy_above = cl;
        S.dmy_at = loc[j];
        found = true;
      }
      cum += tot[j];
      cl += loc[j];
    }
  }
  __syncthreads();
  return DigitCross{S.dsel, S.dabove, S.dcnt, S.dmy_above, S.dmy_at, all};
}

// X selects what is compiled in: KX_PLAIN none of the extended modes, KX_EXT all of them
// (deterministic ties and sorting, hinted sampling, block skipping), KX_BLOCKSKIP block skipping
// alone.  Code a call does not use still costs: the extended instantiation measured ~3 % slower
// than the plain one on plain calls.
enum : int { KX_PLAIN = 0, KX_EXT = 1, KX_BLOCKSKIP = 2 };
template <int X, bool L16>
__global__ void __launch_bounds__(THREADS, 7) gvr_topk_kernel(const Params p) {
  constexpr bool EXT = X == KX_EXT;
  constexpr bool BSK = X != KX_PLAIN;  // block maxima may be given
  constexpr int T = THREADS;
  constexpr int NW = T / 32;
  constexpr int KPT = (MAX_K + T - 1) / T;  // samples per thread at most
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  float4 (*ring)[STAGE_VEC] = reinterpret_cast<float4 (*)[STAGE_VEC]>(smem_raw + SMEM_FIXED);
  const int32_t nst = p.nstage;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t cs = cluster_size();
  const uint32_t rank = cluster_rank();
  const uint32_t row = cluster_id_x();
  const int32_t k = p.k;
  const float qnan = __int_as_float(0x7fffffff);
  // ties at tau go to the smallest window indices (always so when the output is sorted)
  const bool det = EXT && (p.flags & (FLAG_DETERMINISTIC | FLAG_SORTED)) != 0;

  // The ring's barriers are initialized first: the fence that publishes them then overlaps the
  // geometry load instead of delaying the first stage copies.
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < MAX_STAGES; ++s)
      if (s < nst) mbar_init(&S.bar[s], 1);
    mbar_init(&S.hbar, 1);
    mbar_init_fence();
  }

  // Hinted sampling: each CTA of the cluster reads its share of the request's hint row before
  // anything else (it does not depend on the row's length), so the latency overlaps the
  // geometry load; the cluster combines the shares after sampling.
  const int32_t* hints = (EXT && p.mode == MODE_DECODE && p.pre_idx)
                             ? p.pre_idx + int64_t(row / uint32_t(p.next_n)) * p.pre_stride
                             : nullptr;
  int32_t hpos[KPT];
  if (hints) {
    const int hs = (k + int(cs) - 1) / int(cs);  // hints per CTA
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int f = q * T + tid;
      const int i = int(rank) * hs + f;
      hpos[q] = (f < hs && i < k) ? __ldg(hints + i) : -1;
    }
  }

  // ---------------------------------------------------------------- row geometry
  // row_stride < 2^31 and every count below fits in 32 bits.
  const uint32_t stride = uint32_t(p.row_stride);
  uint32_t a = 0, nv = 0;
  if (p.mode == MODE_DECODE) {
    const uint32_t nn = uint32_t(p.next_n);
    const uint32_t req = row / nn;
    const int32_t kv = p.kv_lens[req];
    if (kv >= p.next_n) nv = (uint32_t(kv) - nn + (row - req * nn) + 1u) / uint32_t(p.compress_ratio);
    nv = nv < stride ? nv : stride;
  } else {
    const int32_t ks = p.row_starts[row];
    const int32_t ke = p.row_ends[row];
    const uint32_t s = ks > 0 ? uint32_t(ks) : 0u;
    const uint32_t e = ke > 0 ? (uint32_t(ke) < stride ? uint32_t(ke) : stride) : 0u;
    a = s < stride ? s : stride;
    nv = e > a ? e - a : 0u;
  }
  const float* rowp = p.logits + int64_t(row) * p.row_stride;
  int32_t* out = p.indices + int64_t(row) * k;
  float* outv = p.values ? p.values + int64_t(row) * k : nullptr;
  int32_t* stats = (p.row_stats && rank == 0 && tid == 0) ? p.row_stats + 4 * int64_t(row) : nullptr;

  // ---------------------------------------------------------------- short row: identity
  if (nv <= uint32_t(k)) {
    for (int i = int(rank) * T + tid; i < k; i += int(cs) * T) {
      out[i] = uint32_t(i) < nv ? i : -1;
      if (outv) outv[i] = uint32_t(i) < nv ? rowp[a + i] : -FLT_MAX;
    }
    if (stats) {
      stats[0] = PATH_SHORT;
      stats[1] = stats[2] = stats[3] = 0;
    }
    return;
  }

  // ---------------------------------------------------------------- this CTA's stages
  // Vectors are 16-byte aligned float4s from the aligned column at or below the window start:
  // vector g holds window positions 4g - lead .. 4g + 3 - lead.  The first `lead` lanes of
  // vector 0 and the lanes past the window end in the partial last vector are masked.  The row
  // is cut into stages of STAGE_VEC vectors dealt round-robin to the cluster's CTAs (stage s to
  // rank s % cs), so every CTA sees the whole row evenly, however the scores drift with position.
  const int32_t lead = int32_t(a & 3u);
  const float* base = rowp + (a - uint32_t(lead));
  const int32_t span = lead + int32_t(nv);
  const int32_t ffull = span >> 2;        // whole vectors inside [col0, window end)
  const int32_t tailn = span & 3;         // in-window scalars of the partial last vector
  const int32_t nvec = ffull + (tailn ? 1 : 0);
  const int32_t nrow_stages = (nvec + STAGE_VEC - 1) / STAGE_VEC;
  const int32_t nstages = int32_t(rank) < nrow_stages
                              ? (nrow_stages - int32_t(rank) + int32_t(cs) - 1) / int32_t(cs)
                              : 0;
  auto stage_first = [&](int32_t s) -> int32_t {  // first vector of this CTA's s-th stage
    return (int32_t(rank) + s * int32_t(cs)) * STAGE_VEC;
  };

  // ---------------------------------------------------------------- streaming ring
  // The CTA's stages of every pass go through the ring in order; the ring position (slot,
  // mbarrier phase) advances by one per stage.  Thread 0 refills a slot after all threads have
  // left it.
  bool late = false;
  auto stage_full = [&](int32_t s) -> int32_t {  // whole vectors of stage s (bulk-copied)
    const int32_t c0 = stage_first(s);
    const int32_t c1 = c0 + STAGE_VEC < nvec ? c0 + STAGE_VEC : nvec;
    const int32_t fe = c1 < ffull ? c1 : ffull;
    return fe > c0 ? fe - c0 : 0;
  };
  // Every stage completes exactly one phase of its slot's barrier, even a stage with no whole
  // vector (only the partial tail), so slot phases stay in step with the ring position.
  auto issue_stage = [&](int32_t s, uint32_t slot) {  // one thread per stage
    const int32_t nfull = stage_full(s);
    if (nfull > 0) {
      mbar_arrive_expect_tx(&S.bar[slot], uint32_t(nfull) * 16u);
      bulk_copy_g2s(&ring[slot][0], base + 4 * size_t(stage_first(s)), uint32_t(nfull) * 16u,
                    &S.bar[slot]);
    } else {
      mbar_arrive(&S.bar[slot]);
    }
  };
  // One pass over this CTA's stages: visit(slot, c0) once per stage, after the stage has landed
  // in ring slot `slot`; c0 is the row vector index of the stage's first vector.  All threads
  // call visit the same number of times, so visitors may use warp collectives.  The ring
  // position (slot, phase) of the next stage to consume carries over from pass to pass.
  // A share that fits in the ring stays resident after its first pass: later passes reuse the
  // same slots (their barriers' phases are already complete) instead of copying it again.
  const bool ring_resident = nstages <= nst;
  bool loaded = false;
  uint32_t rslot = 0, rphase = 0;
  // A CTA whose wait gave up (S.tout, set once every thread has seen it) visits no more stages:
  // its row's indices become -2 at the end, and every later pass returns at once.  At the moment
  // it gives up it issues no more refills and waits (bounded) for the copies already in flight,
  // so none is still writing into its shared memory when it moves on or exits.
  // nlim < nstages: only the first nlim stages (all primed, none refilled).
  auto stream_pass = [&](bool primed, auto&& visit, int32_t nlim = -1) {
    if (nlim < 0) nlim = nstages;
    if (S.tout) return;  // CTA-uniform: written before a barrier that every thread has passed
    if (warp == 0 && !primed && !(ring_resident && loaded))
      for (int32_t s = lane; s < nst && s < nlim; s += 32) {  // nst <= 16: one pass of lanes
        const uint32_t sl = rslot + uint32_t(s);
        issue_stage(s, sl < uint32_t(nst) ? sl : sl - uint32_t(nst));
      }
    uint32_t slot = rslot, ph = rphase;
    for (int32_t s = 0; s < nlim; ++s) {
      if (!mbar_wait_bounded(&S.bar[slot], ph, WAIT_LIMIT_NS)) {
        mbar_wait_bounded(&S.bar[slot], ph, WAIT_LIMIT_NS);  // let copies land
        late = true;
      }
      visit(slot, stage_first(s));
      // refill this slot once every thread is done with it, unless some thread gave up waiting
      const bool refill = s + nst < nlim;
      if (refill ? __syncthreads_or(late) : false) {
        // drain: the stages after this one that are already in flight (no refill was issued
        // for this slot), each waited for once, with the same bound
        uint32_t dsl = slot, dph = ph;
        for (int32_t d = s + 1; d < nlim && d < s + nst; ++d) {
          if (++dsl == uint32_t(nst)) {
            dsl = 0;
            dph ^= 1u;
          }
          mbar_wait_bounded(&S.bar[dsl], dph, WAIT_LIMIT_NS);
        }
        late = true;
        break;
      }
      if (refill && tid == 0) issue_stage(s + nst, slot);
      if (++slot == uint32_t(nst)) {
        slot = 0;
        ph ^= 1u;
      }
    }
    if (!ring_resident) {
      rslot = slot;
      rphase = ph;
    }
    loaded = true;
    if (__syncthreads_or(late) && tid == 0) S.tout = 1;
    __syncthreads();  // S.tout is read by the next pass
  };
  // The i-th vector of this thread in the stage at (slot, c0): its share index g, its values
  // and the 4-bit mask of its in-window lanes (0 past the share).
  auto stage_vec = [&](uint32_t slot, int32_t c0, int i, int32_t& g, float4& v) -> uint32_t {
    const int32_t f = i * T + tid;
    g = c0 + f;
    v = f4_zero();
    if (g >= nvec) return 0u;
    uint32_t lanes = 0xFu;
    if (g < ffull) {
      v = ring[slot][f];
    } else {
      v = S.tail;
      lanes = (1u << tailn) - 1u;
    }
    if (g == 0) lanes &= (0xFu << lead) & 0xFu;
    return lanes;
  };
  // Score j (bit j = 4i + l of a stage mask) of this thread in the stage at (slot, c0).
  auto stage_score = [&](uint32_t slot, int32_t c0, int j) -> float {
    const int32_t f = (j >> 2) * T + tid;
    if (c0 + f >= ffull) return f4_get(S.tail, j & 3);
    return reinterpret_cast<const float*>(&ring[slot][0])[4 * f + (j & 3)];
  };
  // Per-lane walk of one stage for the rarely taken passes: f(e, g, valid, l) for every lane of
  // every vector slot of this thread (warp-uniform call count).
  auto each_lane = [&](uint32_t slot, int32_t c0, auto&& f) {
#pragma unroll
    for (int i = 0; i < VPS; ++i) {
      int32_t g;
      float4 v;
      const uint32_t lanes = stage_vec(slot, c0, i, g, v);
#pragma unroll
      for (int l = 0; l < 4; ++l) f(f4_get(v, l), g, ((lanes >> l) & 1u) != 0, l);
    }
  };
  // The same per-lane walk as stream_pass + each_lane, reading the share straight from global
  // memory (no ring): f(e, g, valid, l) for every lane of every vector slot, stage by stage, two
  // stages' loads in flight at a time.  For a pass that must leave the ring alone.
  auto global_pass = [&](auto&& f) {
    const float4* const vbase = reinterpret_cast<const float4*>(base);
    for (int32_t s0 = 0; s0 < nstages; s0 += 2) {
      float4 v[2][VPS];
      uint32_t ln[2][VPS];
      int32_t gg[2][VPS];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int i = 0; i < VPS; ++i) {
          const int32_t g = (s0 + q < nstages) ? stage_first(s0 + q) + i * T + tid : nvec;
          gg[q][i] = g;
          v[q][i] = g < ffull ? __ldg(vbase + g) : S.tail;
          uint32_t lanes = g < ffull ? 0xFu : (g < nvec ? (1u << tailn) - 1u : 0u);
          if (g == 0) lanes &= (0xFu << lead) & 0xFu;
          ln[q][i] = lanes;
        }
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (s0 + q < nstages)  // CTA-uniform
#pragma unroll
          for (int i = 0; i < VPS; ++i)
#pragma unroll
            for (int l = 0; l < 4; ++l) f(f4_get(v[q][i], l), gg[q][i], ((ln[q][i] >> l) & 1u) != 0, l);
    }
  };
  // The list: LCAP scores, then their window indices (int32) or, compact, their positions in
  // this CTA's share (16 bits: stage of the share * 1024 + offset in the stage).
  constexpr int LCAP = L16 ? LIST_CAP16 : LIST_CAP;
  constexpr int LSEG = LCAP / NW;  // each warp appends to its own segment
  const int lcs = __ffs(int(cs)) - 1;  // cs is a power of two
  auto share_to_window = [&](uint32_t sp) -> int32_t {
    return (int32_t(rank) + (int32_t(sp >> 10) << lcs)) * (4 * STAGE_VEC) + int32_t(sp & 1023u) - lead;
  };
  // Index field of the entry for the score at row vector g, lane l (g inside this CTA's share).
  auto list_key = [&](int32_t g, int l) -> uint32_t {
    if constexpr (L16)
      return (uint32_t((g / STAGE_VEC - int32_t(rank)) >> lcs) << 10) + uint32_t(g % STAGE_VEC) * 4u + uint32_t(l);
    else
      return uint32_t(4 * g + l - lead);
  };
  auto list_val = [&](uint32_t at) -> float {
    if constexpr (L16) return S.list_v16[at];
    else return S.list_v[at];
  };
  auto list_put = [&](uint32_t at, float v, uint32_t key) {
    if constexpr (L16) {
      S.list_v16[at] = v;
      S.list_p16[at] = uint16_t(key);
    } else {
      S.list_v[at] = v;
      S.list_j[at] = int32_t(key);
    }
  };
  auto list_keyat = [&](uint32_t at) -> uint32_t {
    if constexpr (L16) return S.list_p16[at];
    else return uint32_t(S.list_j[at]);
  };
  auto list_window = [&](uint32_t at) -> int32_t {
    if constexpr (L16) return share_to_window(S.list_p16[at]);
    else return S.list_j[at];
  };
  // Walk of this CTA's list (every warp segment): f(value, window index, valid), warp-collective
  // with a CTA-uniform trip count.  Only valid once every segment held its scores.
  auto each_listed = [&](auto&& f) {
    uint32_t pre[NW + 1];  // segment starts in the concatenated list
    pre[0] = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) pre[w + 1] = pre[w] + S.list_n[w];
    for (uint32_t b0 = 0; b0 < pre[NW]; b0 += T) {
      const uint32_t i = b0 + tid;
      const bool in = i < pre[NW];
      uint32_t at = i;  // slot of entry i: its segment's base plus its offset in the segment
#pragma unroll
      for (int w = 1; w < NW; ++w)
        if (i >= pre[w]) at = uint32_t(w * LSEG) + (i - pre[w]);
      f(in ? list_val(at) : 0.f, in ? list_window(at) : 0, in);
    }
  };
  // Rank 0, block-collective: reorder out[0..k) (and the values) by (value desc, index asc), the
  // order of the plain definition.  k is a power of two; the 64-bit sort keys (inverted order
  // key, index) live in the histogram / list / ring area, which no CTA uses any more.
  auto sort_output = [&]() {
    uint64_t* sk = reinterpret_cast<uint64_t*>(&S.hist[0]);
    __syncthreads();
    for (int i = tid; i < k; i += T) {
      const int32_t j = __ldcg(out + i);  // written by every CTA of the cluster
      const float v = uint32_t(j) < nv ? __ldg(rowp + a + j) : -INFINITY;
      sk[i] = (uint64_t(~order_key(v)) << 32) | uint32_t(j);
    }
    __syncthreads();
    for (int kk = 2; kk <= k; kk <<= 1)  // bitonic network, ascending
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int i = tid; i < k; i += T) {
          const int l = i ^ jj;
          if (l > i) {
            const uint64_t x = sk[i], y = sk[l];
            if ((x > y) == ((i & kk) == 0)) {
              sk[i] = y;
              sk[l] = x;
            }
          }
        }
        __syncthreads();
      }
    for (int i = tid; i < k; i += T) {
      const int32_t j = int32_t(uint32_t(sk[i]));
      out[i] = j;
      if (outv) outv[i] = uint32_t(j) < nv ? __ldg(rowp + a + j) : -FLT_MAX;
    }
  };
  // After a cluster barrier: tell rank 0 that this CTA gave up waiting (rank 0 marks the row).
  auto report_timeout = [&]() {
    if (tid == 0 && S.tout) dsmem_st_u32(dsmem_map(smem_u32(&S.err), 0), 1u);
  };

  // ---------------------------------------------------------------- guess: block64 sample
  const uint32_t nsamp = sample_count(uint32_t(k), nv, L16 ? 16u : 8u);
  const uint32_t nblk = nsamp >> 6;
  // Start of run b = floor(b (nv - 64) / (nblk - 1)), one run per lane (nblk <= 32), with no
  // 64-bit arithmetic: b (nv - 64) = b sq (nblk - 1) + b sr.
  const uint32_t sq = (nv - 64u) / (nblk - 1u), sr = (nv - 64u) % (nblk - 1u);
  const uint32_t run_start = uint32_t(lane) * sq + (uint32_t(lane) * sr) / (nblk - 1u);
  float sv[KPT];
#pragma unroll
  for (int q = 0; q < KPT; ++q) {  // the 64 samples of a run are 64 consecutive threads' slots
    const uint32_t i = uint32_t(q * T + tid);
    const uint32_t blk = i >> 6;
    const uint32_t s = __shfl_sync(FULL_MASK, run_start, blk & 31u);
    sv[q] = i < nsamp ? __ldg(rowp + a + s + (i & 63u)) : qnan;
  }
  // Hinted sampling adds the k scores at the request's previous selection.  Any content is
  // accepted: positions outside [0, nv) (the -1 pad, stale or garbage entries) are skipped and
  // duplicates only repeat a score, so exactness never depends on the hints.
  float sh[KPT];
  if (hints) {
#pragma unroll
    for (int q = 0; q < KPT; ++q) sh[q] = uint32_t(hpos[q]) < nv ? __ldg(rowp + a + uint32_t(hpos[q])) : qnan;
  }
  // Block-skip rows (block maxima given) may read only the blocks that can reach the floor in
  // the first pass; their first ring stages are staged like every row's (the samples decide
  // later whether skipping pays), and are read whole.
  const float* bmax_row =
      (BSK && p.mode == MODE_DECODE && p.block_max) ? p.block_max + int64_t(row) * p.bmax_stride : nullptr;
  // The first ring stages go in flight right behind the samples, one lane of warp 0 per stage.
  if (warp == 0)
    for (int32_t s = lane; s < nst && s < nstages; s += 32) issue_stage(s, uint32_t(s));
  // Zero the counters while the samples are in flight (global loads are not waited for here).
  static_assert((NB + 4) % 4 == 0, "histograms are cleared as 16-byte vectors");
  for (int i = tid; i < (NB + 4) / 4; i += T) {
    reinterpret_cast<uint4*>(S.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(S.tot)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) {
    for (int w = 0; w < NW; ++w) S.list_n[w] = 0;
    S.ctr_win = S.ctr_cand = S.ctr_rwin = S.ctr_rtie = 0;
    S.gctr_above = S.gctr_cand = 0;
    S.rc_win = S.rc_tie = 0;
    S.tout = S.err = 0;
    S.unlisted = 0;
    S.relist_n = S.relist_bad = 0;
    S.hk_min = S.kmin_loc = 0xffffffffu;
    S.hk_max = S.kmax_loc = 0u;
    S.hlisted = 0;
    S.rec_n = S.saved = 0;  // the block-skip gate's counts, before their own uses
    S.end_hits = S.nbr_hits = 0;
    S.cross = Crossing{};
    S.dsel = S.dabove = S.dcnt = 0;
  }
  if (tid == 32) {  // the partial last vector is read with scalar loads, never past the window
    S.tail = make_float4(qnan, qnan, qnan, qnan);
    if (tailn && (ffull / STAGE_VEC) % int32_t(cs) == int32_t(rank)) {
      const float* q = base + 4 * size_t(ffull);
      S.tail = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
    }
  }
  float lmin = INFINITY, lmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    if (isfinite(sv[q])) {
      lmin = fminf(lmin, sv[q]);
      lmax = fmaxf(lmax, sv[q]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lmin = fminf(lmin, __shfl_xor_sync(FULL_MASK, lmin, o));
    lmax = fmaxf(lmax, __shfl_xor_sync(FULL_MASK, lmax, o));
  }
  // Hinted: the largest finite hinted score widens GMAX (the hints hold the row's top), and the
  // smallest hinted score with the count of in-window hints can raise the floor below.
  if (hints) {
    float hmin = INFINITY, hmax = -INFINITY;
    uint32_t hcnt = 0;
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      if (!isnan(sh[q])) {
        hmin = fminf(hmin, sh[q]);
        ++hcnt;
      }
      if (isfinite(sh[q])) hmax = fmaxf(hmax, sh[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      hmin = fminf(hmin, __shfl_xor_sync(FULL_MASK, hmin, o));
      hmax = fmaxf(hmax, __shfl_xor_sync(FULL_MASK, hmax, o));
      hcnt += __shfl_xor_sync(FULL_MASK, hcnt, o);
    }
    if (lane == 0) {
      S.whmin[warp] = hmin;
      S.whmax[warp] = hmax;
      S.whcnt[warp] = hcnt;
    }
  }
  if (lane == 0) {
    S.wmin[warp] = lmin;
    S.wmax[warp] = lmax;
  }
  __syncthreads();
  if (hints && tid == 0) {  // this CTA's share, published by the barrier below
    float hmin = INFINITY, hmax = -INFINITY;
    uint32_t hcnt = 0;
    for (int w = 0; w < NW; ++w) {
      hmin = fminf(hmin, S.whmin[w]);
      hmax = fmaxf(hmax, S.whmax[w]);
      hcnt += S.whcnt[w];
    }
    S.hpart_min = hmin;
    S.hpart_max = hmax;
    S.hpart_cnt = hcnt;
  }
  // Every CTA's totals and rank 0's counters are now zero; no CTA of the cluster adds to them
  // before it has waited on this (split) barrier, right before its first remote update.  The
  // bulk adds that land in the totals go through the async proxy, so the zeros are fenced
  // for it first.
  fence_proxy_async_smem();
  cluster_arrive();
  bool init_waited = false;
  auto wait_init = [&]() {
    if (!init_waited) {
      cluster_wait();
      init_waited = true;
    }
  };
  auto csync = [&]() {
    wait_init();
    cluster_sync();
  };
  float gmin = INFINITY, gmax = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    gmin = fminf(gmin, S.wmin[w]);
    gmax = fmaxf(gmax, S.wmax[w]);
  }
  if (hints) {  // every CTA's share of the hints, read from the cluster after the barrier
    wait_init();
    if (warp == 0) {
      float hmin = INFINITY, hmax = -INFINITY;
      uint32_t hcnt = 0;
      if (uint32_t(lane) < cs) {
        hmin = __uint_as_float(dsmem_ld_u32(dsmem_map(smem_u32(&S.hpart_min), uint32_t(lane))));
        hmax = __uint_as_float(dsmem_ld_u32(dsmem_map(smem_u32(&S.hpart_max), uint32_t(lane))));
        hcnt = dsmem_ld_u32(dsmem_map(smem_u32(&S.hpart_cnt), uint32_t(lane)));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        hmin = fminf(hmin, __shfl_xor_sync(FULL_MASK, hmin, o));
        hmax = fmaxf(hmax, __shfl_xor_sync(FULL_MASK, hmax, o));
        hcnt += __shfl_xor_sync(FULL_MASK, hcnt, o);
      }
      if (lane == 0) {
        S.hagg_min = hmin;
        S.hagg_max = hmax;
        S.hagg_cnt = hcnt;
      }
    }
    __syncthreads();
    gmax = fmaxf(gmax, S.hagg_max);
  }
  gmin = __fadd_rn(gmin, 0.0f);  // -0 -> +0, so every CTA holds the same bits
  const bool bracket_ok = isfinite(gmin) && isfinite(gmax) && gmin < gmax;

  int path = PATH_REFINE;
  if (p.flags & FLAG_FORCE_RESCUE) path = PATH_RESCUE_FORCED;
  else if (!bracket_ok) path = PATH_RESCUE_BRACKET;

  // Block-skip gate: skipping pays only while very few blocks reach the floor (the skipping
  // pass reads its blocks with plain loads, far fewer bytes in flight than the ring's bulk
  // copies).  The block64 samples are runs of two 32-score halves spread over the row; the
  // share of the interior halves with a sample at or above the floor estimates the share of
  // blocks the skipping pass would still read (the same in every CTA of the row: same samples,
  // same floor).  Above 1/16 the row takes the staged pass.  Counted before the floor's
  // barrier, read after it.
  bool skip_blocks = false;
  uint32_t floor_want = 0;  // samples at or above the floor (0: no floor)
  float sc = 0.f;
  float thr = -INFINITY;  // floor: scores >= thr are counted (and listed) in the first pass
  int fpart = -1;         // bin(thr): the one partially counted bin; -1 = no floor
  if (path == PATH_REFINE) {
    sc = __fdiv_rn(float(NB), __fsub_rn(gmax, gmin));
    if (!(p.flags & FLAG_NO_FLOOR)) {
      // mu = k*nsamp/nv samples are expected above tau (a Poisson count); keep mu + 3 sqrt(mu)
      // + 6 above the floor.  A second pass is then rare enough per row (below 1e-4 for every mu
      // of the workloads) that a batch of hundreds of rows seldom has one: the launch waits for
      // its slowest row, so the margin is sized for the batch, not for the single row.
      const float mu = float(k) * float(nsamp) / float(nv);
      const float want_f = mu + 3.0f * sqrtf(mu) + 6.0f;
      const uint32_t want = want_f < float(nsamp) ? uint32_t(want_f) : nsamp;
      floor_want = want;
      // The samples' own histogram on the same bins (in this CTA's private counts, cleared
      // again below): the floor is the lower edge of the bin where `want` samples are reached.
#pragma unroll
      for (int q = 0; q < KPT; ++q)
        if (!isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
      __syncthreads();
      int fb = suffix_cross<T>(S, S.hist, want);
      // A far outlier sample stretches every bin, and with them the floor's bin (more scores
      // listed) and the crossing bin (more candidates).  When mu is large enough that the r-th
      // largest sample, r = mu - 4 sqrt(mu), lies above tau all but surely, the bins end at the
      // top of that sample's bin instead: the scores above it clamp into the top bin, which then
      // holds about (1 - 4 / sqrt(mu)) k of them, all winners, and the floor is found again on
      // the narrower bins.  Only when the floor and that sample sit in the lower half of the
      // bins (a handful of far samples stretched them).  The samples, and so the scale, are the
      // same in every CTA.
      const float rf = mu - 4.0f * sqrtf(mu);
      const int hb = (rf >= 2.0f && fb < NB / 2) ? suffix_cross<T>(S, S.hist, uint32_t(rf)) : -1;
      if (hb >= 0 && hb < NB / 2) {
        const float hi = __fadd_rn(gmin, __fdiv_rn(float(hb + 1), sc));
        sc = __fdiv_rn(float(NB), __fsub_rn(hi, gmin));
        for (int i = tid; i < NB; i += T) S.hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < KPT; ++q)
          if (!isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
        __syncthreads();
        fb = suffix_cross<T>(S, S.hist, want);
      }
      // Block-concentrated rows (a sink and recent tokens at the row's two ends, hot blocks in
      // between) put the first and the last run on the hot ends: the samples over-represent the
      // top, the floor lands above tau and every such row would count its scores twice.  When
      // the two end runs hold most of the samples at or above the floor's bin while their
      // neighbouring runs hold few, the floor is found again from the interior runs alone (the
      // target scaled to their number) and the lower of the two is kept.  A smooth trend (a
      // position bias) raises the neighbours too and keeps the floor.  Compiled into the
      // block-skip instantiations only (the entry point for attention rows of that shape): the
      // check measured 2-4 % on the plain path's other rows.
      const bool ends_check = BSK && bmax_row && nblk >= 6;
      if (ends_check) {
        uint32_t ec = 0, nc = 0;
#pragma unroll
        for (int q = 0; q < KPT; ++q) {
          if (uint32_t(q * T) >= 128u && uint32_t((q + 1) * T) + 128u <= nsamp) continue;  // no end run here
          const uint32_t i = uint32_t(q * T + tid), run = i >> 6;
          if (i < nsamp && !isnan(sv[q]) && value_bin(sv[q], gmin, sc) >= fb) {
            ec += (run == 0 || run == nblk - 1) ? 1u : 0u;
            nc += (run == 1 || run == nblk - 2) ? 1u : 0u;
          }
        }
        if (ec) atomicAdd(&S.end_hits, ec);
        if (nc) atomicAdd(&S.nbr_hits, nc);
      }
      if (BSK && bmax_row) {
        const float tf = fb > 0 ? __fadd_rn(gmin, __fdiv_rn(float(fb), sc)) : -FLT_MAX;  // the floor
        uint32_t hitq = 0, validq = 0;  // bit q: this warp's 32 samples of slot q reach it / count
#pragma unroll
        for (int q = 0; q < KPT; ++q) {  // the end runs (sink, recent tokens) are left out
          const uint32_t i0 = uint32_t(q * T + 32 * warp);
          hitq |= uint32_t(sv[q] >= tf) << q;
          validq |= uint32_t(i0 >= 64u && i0 + 96u <= nsamp) << q;
        }
        hitq = __reduce_or_sync(FULL_MASK, hitq) & validq;
        if (lane == 0) {
          atomicAdd(&S.rec_n, uint32_t(__popc(hitq)));
          atomicAdd(&S.saved, uint32_t(__popc(validq)));
        }
      }
      auto set_floor = [&]() {  // tid 0
        // any threshold works: bins above bin(t) are complete, bin(t) is partial.  A floor in
        // the lowest bin is -FLT_MAX: every score but -inf (and NaN) is counted and listed, so a
        // row whose finite scores are fewer than k is decided by the first pass (the -inf fill)
        const float t = fb > 0 ? __fadd_rn(gmin, __fdiv_rn(float(fb), sc)) : -FLT_MAX;
        S.vthr = t;
        S.fpart = value_bin(t, gmin, sc);
      };
      if (tid == 0) set_floor();
      for (int i = tid; i < NB / 4; i += T) reinterpret_cast<uint4*>(S.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      if (BSK && bmax_row)
        skip_blocks = (p.flags & FLAG_BLOCKSKIP_ALWAYS) || (S.saved > 0u && 16u * S.rec_n <= S.saved);
      if (ends_check && 3u * S.end_hits >= 2u * want && S.end_hits >= 4u * (S.nbr_hits + 1u)) {
        const uint32_t nint = nsamp - 128u;
        const float mui = float(k) * float(nint) / float(nv);
        const float wi = mui + 3.0f * sqrtf(mui) + 6.0f;
        const uint32_t want_i = wi < float(nint) ? uint32_t(wi) : nint;
#pragma unroll
        for (int q = 0; q < KPT; ++q) {
          const uint32_t i = uint32_t(q * T + tid);
          if (i >= 64u && i + 64u < nsamp && !isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
        }
        __syncthreads();
        const int fbi = suffix_cross<T>(S, S.hist, want_i);
        if (fbi < fb) {
          fb = fbi;
          if (tid == 0) set_floor();
        }
        for (int i = tid; i < NB; i += T) S.hist[i] = 0;
        __syncthreads();
      }
      thr = S.vthr;
      fpart = S.fpart;
      if (hints) {
        // k in-window hints at k distinct positions put at least k scores at or above the
        // smallest hinted score, so a floor there needs no second pass (with fewer distinct
        // positions the second pass still makes the counts exact).
        const float hm = __fadd_rn(S.hagg_min, 0.0f);  // -0 -> +0
        const uint32_t hc = S.hagg_cnt;
        if (hc == uint32_t(k) && hm > thr) {
          thr = hm;
          fpart = value_bin(hm, gmin, sc);
        }
      }
    }
  }

  Crossing cr{};
  int rounds = 0;
  bool listed = false;  // the list holds every score >= thr of this CTA's share
  if (path == PATH_REFINE) {
    // ------------------------------------------------------------ verify: value histogram
    // Pass 1 counts (and lists) the scores >= thr; pass 2, only when the crossing falls in
    // the partial bin or below, counts the rest.
    uint32_t wlist = 0;  // scores this warp has appended (warp-uniform; may exceed LSEG)
    // Dense share: when the floor lets through more of this CTA's scores than its list holds
    // (by the samples' share above it, with a quarter of margin) -- K = 2048 on a window of a
    // few thousand scores -- the list would overflow and the collect read the share again
    // anyway, so the pass only counts from the start: no list slots, no list stores, no walk of
    // the list after the pass.  The list is marked incomplete.  (A floor of -FLT_MAX keeps
    // listing: the -inf fill needs every CTA's list.)
    const bool dense_start = floor_want > 0u && thr > -FLT_MAX &&
                             uint64_t(4u * floor_want) * uint64_t(nstages) * uint64_t(4 * STAGE_VEC) >
                                 uint64_t(5u) * nsamp * uint64_t(LCAP);
    float* const seg_v = (L16 ? S.list_v16 : S.list_v) + warp * LSEG;  // this warp's segment
    int32_t* const seg_j = S.list_j + warp * LSEG;
    uint16_t* const seg_p = S.list_p16 + warp * LSEG;
    {
      // One stage per visit, with no warp collective: a thread with scores >= thr takes list
      // slots for them with one shared-memory atomic on its warp's counter (S.list_n[warp]) and
      // lists them; their bins are counted once the pass is over, from the list.  A thread that
      // finds its warp's segment full lists what still fits and from then on only counts its
      // hits, in a register run of one bin that goes to the histogram when the bin changes (a
      // tie class costs one atomic per thread for the whole pass).  The counter then exceeds
      // the segment, which marks the list incomplete; the counts stay exact either way.
      constexpr int NE = 4 * VPS;
      bool full = dense_start;             // this thread saw its warp's segment full
      if (dense_start && lane == 0) S.list_n[warp] = uint32_t(LSEG) + 1u;  // incomplete, holds nothing
      uint32_t rb = 0xffffffffu, rrun = 0;  // its run of counted hits in bin rb
      float rv = __int_as_float(0x7fffffff);  // the run's last value (NaN: none yet)
      float hv0 = INFINITY, hv1 = -INFINITY;  // smallest / largest of its hits (NaN never hits)
      const int32_t ring_stages = skip_blocks ? (nstages < nst ? nstages : nst) : nstages;
      stream_pass(true, [&](uint32_t slot, int32_t c0) {
        float4 vv[VPS];
        uint32_t lanes;  // bit 4v+l: lane l of this thread's v-th vector is in the window
        if (c0 > 0 && c0 + STAGE_VEC <= ffull) {  // an interior stage: every lane is in
#pragma unroll
          for (int i = 0; i < VPS; ++i) vv[i] = ring[slot][i * T + tid];
          lanes = (1u << NE) - 1u;
        } else {
          lanes = 0;
#pragma unroll
          for (int i = 0; i < VPS; ++i) {
            int32_t g;
            lanes |= stage_vec(slot, c0, i, g, vv[i]) << (4 * i);
          }
        }
        uint32_t bits = 0;  // bit 4v+l: lane l of this thread's v-th vector is >= thr
#pragma unroll
        for (int v = 0; v < VPS; ++v)
          bits |= (uint32_t(vv[v].x >= thr) | (uint32_t(vv[v].y >= thr) << 1) | (uint32_t(vv[v].z >= thr) << 2) |
                   (uint32_t(vv[v].w >= thr) << 3))
                  << (4 * v);
        bits &= lanes;
        if (!bits) return;
        if (!full) {
          const uint32_t nb = uint32_t(__popc(bits));
          uint32_t at = atomicAdd(&S.list_n[warp], nb);
          const bool fits = at + nb <= uint32_t(LSEG);
          const uint32_t end = fits ? at + nb : uint32_t(LSEG);
          for (; at < end; ++at) {  // list (all of them, or what still fits)
            const int j = __ffs(bits) - 1;
            bits &= bits - 1u;
            seg_v[at] = stage_score(slot, c0, j);
            if constexpr (L16)
              seg_p[at] = uint16_t(list_key(c0 + tid, 0) + uint32_t(j >> 2) * (4 * T) + uint32_t(j & 3));
            else
              seg_j[at] = 4 * (c0 + tid) - lead + (j >> 2) * (4 * T) + (j & 3);
          }
          if (fits) return;
          full = true;
        }
        uint32_t same = 0;  // hits equal to the run's last value: same bin, no bin arithmetic
#pragma unroll
        for (int j = 0; j < NE; ++j) same |= uint32_t(f4_get(vv[j >> 2], j & 3) == rv) << j;
        if ((bits & ~same) == 0u) {
          rrun += uint32_t(__popc(bits));
          return;
        }
        // Otherwise every hit of the stage is added on its own, with no dependence between them
        // (all bins first, then one atomic per hit); the stage's first hit becomes the run's value
        // for the stages after (a tie class then takes the shortcut above).
        uint32_t bj[NE];
#pragma unroll
        for (int j = 0; j < NE; ++j) bj[j] = uint32_t(value_bin(f4_get(vv[j >> 2], j & 3), gmin, sc));
#pragma unroll
        for (int j = 0; j < NE; ++j)
          if ((bits >> j) & 1u) {
            const float e = f4_get(vv[j >> 2], j & 3);
            atomicAdd(&S.hist[bj[j]], 1u);
            hv0 = fminf(hv0, e);
            hv1 = fmaxf(hv1, e);
          }
        if (rrun) atomicAdd(&S.hist[rb], rrun);
        const int jf = __ffs(bits) - 1;
        rv = stage_score(slot, c0, jf);
        rb = uint32_t(value_bin(rv, gmin, sc));
        rrun = 0;
      }, ring_stages);
      if (rrun) atomicAdd(&S.hist[rb], rrun);
      __syncwarp();
      wlist = S.list_n[warp];
      // The listed hits' bins, counted once per list entry (the entries past a full segment
      // were counted during the pass).
      const uint32_t nl = dense_start ? 0u : (wlist < uint32_t(LSEG) ? wlist : uint32_t(LSEG));
      for (uint32_t i = uint32_t(lane); i < nl; i += 32u) {
        const float e = seg_v[i];
        atomicAdd(&S.hist[value_bin(e, gmin, sc)], 1u);
        hv0 = fminf(hv0, e);
        hv1 = fmaxf(hv1, e);
      }
      // this CTA's key bounds of the scores >= thr (for a row whose scores >= thr are one value)
      uint32_t hk0 = hv0 <= hv1 ? order_key(hv0) : 0xffffffffu, hk1 = hv0 <= hv1 ? order_key(hv1) : 0u;
      hk0 = __reduce_min_sync(FULL_MASK, hk0);
      hk1 = __reduce_max_sync(FULL_MASK, hk1);
      if (lane == 0 && hk0 <= hk1) {
        atomicMin(&S.kmin_loc, hk0);
        atomicMax(&S.kmax_loc, hk1);
      }
    }
    if (skip_blocks) {
      // ---------------------------------------------------------- block-skip first pass
      // ("Block-skip fast path for self-sampling GVR top-K decode", opt-in row pass): a block
      // of 32 scores whose bound is below the floor holds no score the first pass counts, so
      // only the surviving blocks are read, with plain coalesced loads (one block per warp
      // load, up to 8 in flight per warp).  The counts and lists equal those of the full pass.
      const int64_t wend = int64_t(a) + nv;  // decode: a = 0, the window is [0, nv)
      // The stages the ring did not hold, one warp each; the warp's list continues after the
      // ring part's entries (whose bins are already counted).
      for (int32_t s = nst + warp; s < nstages; s += NW) {
        const int64_t colst = 4 * int64_t(stage_first(s));  // first column (a multiple of 1024)
        const int64_t bi = (colst >> 5) + lane;              // this lane's block
        const bool inwin = bi * 32 < wend;
        const float bm = inwin ? __ldg(bmax_row + bi) : -INFINITY;
        unsigned surv = __ballot_sync(FULL_MASK, inwin && !(bm < thr));  // NaN bounds survive
        while (surv) {
          int32_t blk[8];
          float v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            blk[q] = surv ? __ffs(surv) - 1 : -1;
            surv &= surv - 1u;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int64_t col = colst + 32 * blk[q] + lane;
            v[q] = (blk[q] >= 0 && col < wend) ? __ldg(rowp + col) : -INFINITY;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (blk[q] < 0) break;  // warp-uniform
            const int64_t col = colst + 32 * blk[q] + lane;
            const bool hit = col < wend && v[q] >= thr;
            const unsigned hm = __ballot_sync(FULL_MASK, hit);
            if (!hm) continue;
            const uint32_t at = wlist + uint32_t(__popc(hm & lanemask_lt()));
            wlist += uint32_t(__popc(hm));
            if (hit) atomicAdd(&S.hist[value_bin(v[q], gmin, sc)], 1u);
            if (hit && at < uint32_t(LSEG)) {
              seg_v[at] = v[q];
              if constexpr (L16) seg_p[at] = uint16_t(s * 1024 + 32 * blk[q] + lane);
              else seg_j[at] = int32_t(col - a);
            }
          }
        }
      }
    }
    // Diagnostics: the first row's rank-0 CTA reports a give-up here, after its first pass has
    // waited for every stage it issued (nothing in flight), to exercise the failure path.
    if ((p.flags & FLAG_DIAG_FAIL_ROW0) && row == 0 && rank == 0 && tid == 0) S.tout = 1;
    if (lane == 0) S.list_n[warp] = wlist;
    __syncthreads();
    listed = true;
#pragma unroll
    for (int w = 0; w < NW; ++w) listed = listed && S.list_n[w] <= uint32_t(LSEG);
    if (L16) listed = listed && nstages <= LIST_MAX_STAGES;  // positions fit 16 bits
    rounds = 1;
    // Push this CTA's counts of bins [b0, b1] into every CTA's totals (fire-and-forget).
    auto push = [&](int b0, int b1) {
      wait_init();
      for (int b = b0 + tid; b <= b1; b += T) {
        const uint32_t v = S.hist[b];
        if (v) {
          const uint32_t local = smem_u32(&S.tot[b]);
          for (uint32_t c = 0; c < cs; ++c) dsmem_red_add(dsmem_map(local, c), v);
        }
      }
    };
    // The counts of bins >= the floor's bin go to every CTA of the cluster.  A narrow range
    // (the usual case: the floor a few hundred bins below the sampled maximum) goes as bulk
    // adds, one per destination from a 16-byte boundary (the bins below the floor are zero
    // here), with the list flag in hist[NB]; each CTA's barrier counts the bytes of all of them
    // (the floor is cluster-uniform, so every CTA expects the same count) and no cluster
    // barrier is needed.  A wide range -- a far outlier stretched the bins, few of them are
    // occupied -- goes bin by bin, only the occupied ones, then a cluster barrier.
    // This CTA's key bounds and listed count go to every CTA, one thread per destination, after
    // the counts are on their way (read after a later cluster barrier, only by the rescue).
    auto publish_bounds = [&]() {
      if (!bmax_row && uint32_t(tid) < cs) {
        uint32_t lc = 0;
        if (!dense_start) {
#pragma unroll
          for (int w = 0; w < NW; ++w) lc += min(S.list_n[w], uint32_t(LSEG));
        }
        const uint32_t c = uint32_t(tid);
        if (S.kmin_loc <= S.kmax_loc) {
          dsmem_red_min(dsmem_map(smem_u32(&S.hk_min), c), S.kmin_loc);
          dsmem_red_max(dsmem_map(smem_u32(&S.hk_max), c), S.kmax_loc);
        }
        if (lc) dsmem_red_add(dsmem_map(smem_u32(&S.hlisted), c), lc);
      }
    };
    const int fb0 = (fpart > 0 ? fpart : 0) & ~3;
    if (NB - fb0 <= BULK_BINS) {
      const uint32_t pbytes = uint32_t(NB + 4 - fb0) * 4u;
      if (tid == 0) S.hist[NB] = listed ? 0u : (rank == 0 ? 1u + UNLISTED_RANK0 : 1u);
      fence_proxy_async_smem();  // the counts, written by this CTA's threads, are read by the bulk copies
      wait_init();               // every CTA's totals are zero and its barrier initialized
      __syncthreads();
      if (tid == 0) {
        for (uint32_t c = 0; c < cs; ++c)
          bulk_reduce_add_u32(dsmem_map(smem_u32(&S.tot[fb0]), c), &S.hist[fb0], pbytes,
                              dsmem_map(smem_u32(&S.hbar), c));
        mbar_arrive_expect_tx(&S.hbar, cs * pbytes);
      }
      publish_bounds();
      if (!mbar_wait_bounded(&S.hbar, 0, WAIT_LIMIT_NS)) late = true;
      if (__syncthreads_or(late) && tid == 0) S.tout = 1;
      if (tid == 0) S.unlisted = S.tot[NB];
    } else {
      push(fpart > 0 ? fpart : 0, NB - 1);
      publish_bounds();
      if (tid == 0 && !listed)
        for (uint32_t c = 0; c < cs; ++c)
          dsmem_red_add(dsmem_map(smem_u32(&S.unlisted), c), rank == 0 ? 1u + UNLISTED_RANK0 : 1u);
      csync();
    }
    report_timeout();
    cr = scan_crossing<T>(S, uint32_t(k));
    if (thr == -FLT_MAX && cr.total < uint32_t(k) && S.unlisted == 0 && !det) {
      // Fewer than k scores are >= -FLT_MAX and every CTA listed all of its own: tau = -inf (NaN
      // aside).  The listed scores are the winners; any k - total of the others fill the rest.
      path = PATH_NEG_INF_FILL;
    } else if (fpart >= 0 && cr.total < uint32_t(k)) {
      // Fewer than k scores reached the floor: count the scores below it, push only these new
      // counts, then scan the complete totals.  (When at least k scores reached the floor, tau
      // is at or above it, and a crossing in the partial floor bin needs no second pass: its
      // candidates are the counted scores, those >= thr.)
      rounds = 2;
      // every CTA has finished reading its totals before new counts arrive, and every bulk add
      // of the first counts (reading hist) has landed
      csync();
      if (tid == 0) {
        S.saved = S.hist[fpart];
        S.hist[fpart] = 0;
      }
      __syncthreads();
      stream_pass(false, [&](uint32_t slot, int32_t c0) {
        each_lane(slot, c0, [&](float e, int32_t, bool valid, int) {
          // most scores hit here, with bins that differ: plain atomics (the hardware merges
          // lanes that share an address) beat aggregating them first
          const bool hit = valid && e < thr;
          if (hit) atomicAdd(&S.hist[value_bin(e, gmin, sc)], 1u);
        });
      });
      push(0, fpart);
      csync();
      report_timeout();
      if (tid == 0) S.hist[fpart] += S.saved;
      __syncthreads();
      cr = scan_crossing<T>(S, uint32_t(k));
    }
    const uint32_t cap = (p.flags & FLAG_ZERO_CAP) ? 0u : uint32_t(CAP);
    if (path == PATH_NEG_INF_FILL) {
      // decided by the first pass
    } else if (cr.total < uint32_t(k))
      path = PATH_RESCUE_OVERFLOW;  // NaN in the window (out of contract)
    else if (cr.m > cap && (p.flags & FLAG_ZERO_CAP || det || rounds != 1 || S.unlisted >= UNLISTED_RANK0 ||
                            cr.m > uint32_t(nst) * RING_CAND))
      // every list complete: the cluster selects among the listed scores
      path = (rounds == 1 && S.unlisted == 0 && !(p.flags & FLAG_STREAM_RESCUE)) ? PATH_REFINE_CLUSTER
                                                                                   : PATH_RESCUE_OVERFLOW;
    // else CAP < m <= (ring stages) * RING_CAND after one pass with rank 0's list complete: rank
    // 0 collects the candidates in its ring, idle since rank 0 does not read the row again (CTAs
    // whose list overflowed read their own share through their own ring), and refines alone
  }
  // Candidates are the scores of the crossing bin that were counted: after one pass, the scores
  // >= thr (this only matters when the crossing is the partial floor bin).
  const float cthr = rounds == 1 ? thr : -INFINITY;

  if (path == PATH_NEG_INF_FILL) {
    // ------------------------------------------------------------ -inf fill
    // Winners: every listed score (total of them, cluster-wide).  Ties: k - total of the other
    // in-window scores, all -inf for a row inside the contract.  Rank 0 hands each CTA a block of
    // winner slots (its listed count) and of tie slots (its unlisted in-window count); a CTA
    // walks its share for ties only until its tie slots are written.
    const uint32_t nwin = cr.total, nties = uint32_t(k) - cr.total;
    uint32_t my_win = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) my_win += S.list_n[w];
    if (tid == 0) {
      uint32_t share = 0;  // in-window scores of this CTA's stages
      for (int32_t st = 0; st < nstages; ++st) {
        const int32_t c0 = stage_first(st), c1 = min(c0 + STAGE_VEC, nvec);
        int32_t n = 4 * (c1 - c0);
        if (c0 == 0) n -= lead;
        if (c1 == nvec && tailn) n -= 4 - tailn;
        share += uint32_t(n);
      }
      S.base_above = dsmem_atom_add(dsmem_map(smem_u32(&S.gctr_above), 0), my_win);
      S.saved = share - my_win;  // this CTA's ties
      S.base_cand = dsmem_atom_add(dsmem_map(smem_u32(&S.gctr_cand), 0), share - my_win);
    }
    __syncthreads();
    const uint32_t wbase = S.base_above, tbase = S.base_cand, my_eq = S.saved;
    each_listed([&](float e, int32_t jw, bool in) {
      const uint32_t ws = warp_alloc_local(&S.ctr_win, in);
      if (in && wbase + ws < nwin) {
        out[wbase + ws] = jw;
        if (outv) outv[wbase + ws] = e;
      }
    });
    const uint32_t my_ties = tbase < nties ? min(my_eq, nties - tbase) : 0u;
    if (my_ties > 0) {
      stream_pass(false, [&](uint32_t slot, int32_t c0) {
        if (S.ctr_cand >= my_ties) return;  // warp-uniform read; the counter only grows
        uint32_t tm = 0;
        each_lane(slot, c0, [&](float e, int32_t g, bool valid, int l) {
          tm |= uint32_t(valid && !(e >= thr)) << (4 * ((g - c0) / T) + l);
        });
        uint32_t ts = warp_alloc_n(&S.ctr_cand, __popc(tm));
        for (uint32_t rest = tm; rest; rest &= rest - 1, ++ts)
          if (ts < my_ties) {
            const int j = __ffs(rest) - 1;
            out[nwin + tbase + ts] = 4 * (c0 + (j >> 2) * T + tid) + (j & 3) - lead;
            if (outv) outv[nwin + tbase + ts] = stage_score(slot, c0, j);
          }
      });
    }
    report_timeout();
    csync();  // rank 0's counters stay alive until every CTA is done with them
    if (rank == 0) {
      const bool failed = S.err || S.tout;
      if (failed)
        for (int i = tid; i < k; i += T) out[i] = -2;
      if (stats) {
        stats[0] = failed ? PATH_DEVICE_ERROR : PATH_NEG_INF_FILL;
        stats[1] = int32_t(nties);
        stats[2] = rounds;
        stats[3] = int32_t(nwin);
      }
    }
    return;
  }

  if (path == PATH_REFINE) {
    // ------------------------------------------------------------ collect
    // Rank 0 hands each CTA a contiguous block of winner slots and of candidate slots.
    if (tid == 0) S.base_above = dsmem_atom_add(dsmem_map(smem_u32(&S.gctr_above), 0), cr.my_above);
    if (tid == 32) S.base_cand = dsmem_atom_add(dsmem_map(smem_u32(&S.gctr_cand), 0), cr.my_cand);
    __syncthreads();
    const int bstar = cr.bin;
    // The candidates go to rank 0's ring, idle from now on: its first stage holds CAP of them
    // (scores, then indices), the whole ring up to nst * RING_CAND when rank 0 reads nothing again.
    // When rank 0 reads its share again in this collect (its list overflowed, or scores below the
    // floor count), its list area is idle instead: up to CAP candidates go there and rank 0
    // streams its share through its ring; more candidates keep the ring and rank 0 reads from
    // global memory.  (Cluster-uniform: the rounds and rank 0's list flag in the pushed counts.)
    const bool big = cr.m > uint32_t(CAP);
    const bool cand_in_list = !big && (rounds != 1 || S.unlisted >= UNLISTED_RANK0);
    const uint32_t ring_cap = uint32_t(nst) * RING_CAND;
    const uint32_t cand_cap = big ? ring_cap : uint32_t(CAP);
    static_assert(sizeof(float) * CAP + sizeof(int32_t) * CAP <= LIST_BYTES, "CAP candidates fit the list area");
    float* const cand_v = cand_in_list ? &S.list_v[0] : reinterpret_cast<float*>(&ring[0][0]);
    int32_t* const cand_j = (cand_in_list ? reinterpret_cast<int32_t*>(&S.list_v[0])
                                          : reinterpret_cast<int32_t*>(&ring[0][0])) + cand_cap;
    const uint32_t rv = dsmem_map(smem_u32(cand_v), 0);
    const uint32_t rj = dsmem_map(smem_u32(cand_j), 0);
    auto place = [&](float e, int32_t jw, bool valid) {  // warp-collective
      const int b = valid ? value_bin(e, gmin, sc) : -1;
      const uint32_t ws = warp_alloc_local(&S.ctr_win, b > bstar);
      if (b > bstar) {
        const uint32_t slot = S.base_above + ws;
        if (slot < uint32_t(k)) {  // always true: counts match the histogram's
          out[slot] = jw;
          if (outv) outv[slot] = e;
        }
      }
      const uint32_t cslot = warp_alloc_local(&S.ctr_cand, b == bstar);
      if (b == bstar) {
        const uint32_t c = S.base_cand + cslot;
        if (c < cand_cap) {  // always true: m fits the buffer on this path
          dsmem_st_u32(rv + 4u * c, __float_as_uint(e));
          dsmem_st_u32(rj + 4u * c, uint32_t(jw));
        }
      }
    };
    if (!(rounds == 1 && listed)) rounds += 10;  // diagnostics: collect read the share again
    if (rounds == 1 && listed) {
      // From the list, with no warp collective: each thread counts its entries' winners and
      // candidates, takes their slots with one shared atomic per kind, then writes them.
      uint32_t pre[NW + 1];  // segment starts in the concatenated list
      pre[0] = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) pre[w + 1] = pre[w] + S.list_n[w];
      auto slot_of = [&](uint32_t i) {  // entry i: its segment's base plus its offset in it
        uint32_t at = i;
#pragma unroll
        for (int w = 1; w < NW; ++w)
          if (i >= pre[w]) at = uint32_t(w * LSEG) + (i - pre[w]);
        return at;
      };
      uint32_t nw = 0, nc = 0;
      for (uint32_t i = tid; i < pre[NW]; i += T) {
        const int b = value_bin(list_val(slot_of(i)), gmin, sc);
        nw += b > bstar ? 1u : 0u;
        nc += b == bstar ? 1u : 0u;
      }
      if (nw | nc) {
        uint32_t wat = nw ? S.base_above + atomicAdd(&S.ctr_win, nw) : 0u;
        uint32_t cat = nc ? S.base_cand + atomicAdd(&S.ctr_cand, nc) : 0u;
        for (uint32_t i = tid; i < pre[NW]; i += T) {
          const uint32_t at = slot_of(i);
          const float e = list_val(at);
          const int b = value_bin(e, gmin, sc);
          if (b > bstar) {
            if (wat < uint32_t(k)) {  // always true: counts match the histogram's
              out[wat] = list_window(at);
              if (outv) outv[wat] = e;
            }
            ++wat;
          } else if (b == bstar) {
            if (cat < cand_cap) {  // always true: m fits the buffer on this path
              dsmem_st_u32(rv + 4u * cat, __float_as_uint(e));
              dsmem_st_u32(rj + 4u * cat, uint32_t(list_window(at)));
            }
            ++cat;
          }
        }
      }
    } else {  // the list overflowed or scores below the floor count: read the share again
      if (warp == 0) {
        const float t = bstar > 0 ? floor_value(bstar, gmin, sc) : -INFINITY;
        const float t1 = bstar < NB - 1 ? floor_value(bstar + 1, gmin, sc) : INFINITY;
        if (lane == 0) {
          S.vthr = t;
          S.vthr1 = t1;
        }
      }
      __syncthreads();
      const float tb = S.vthr;  // scores >= tb are exactly those in bins >= b*
      const float tb1 = S.vthr1;  // ... and >= tb1 those in bins > b* (none when b* is the top bin)
      const bool top = bstar == NB - 1;
      auto visit = [&](float e, int32_t g, bool valid, int l) {
        const bool hit = valid && e >= tb && e >= cthr;
        if (__any_sync(FULL_MASK, hit)) place(e, 4 * g + l - lead, hit);
      };
      // A staged share, with no warp collective: each thread marks its winners and candidates of
      // the stage, takes their slots with one shared atomic per kind, and writes them.  (A warp
      // prefix of the counts, one atomic per warp, measured slower even on dense rows.)
      auto collect_stage = [&](uint32_t slot, int32_t c0) {
        uint32_t wm = 0, cm = 0;
#pragma unroll
        for (int i = 0; i < VPS; ++i) {
          int32_t g;
          float4 v;
          const uint32_t ln = stage_vec(slot, c0, i, g, v);
#pragma unroll
          for (int l = 0; l < 4; ++l) {
            const float e = f4_get(v, l);
            if (((ln >> l) & 1u) && e >= tb && e >= cthr) {  // bins are monotone: compares only
              const bool above = !top && e >= tb1;
              wm |= uint32_t(above) << (4 * i + l);
              cm |= uint32_t(!above) << (4 * i + l);
            }
          }
        }
        auto window_of = [&](int j) { return 4 * (c0 + (j >> 2) * T + tid) + (j & 3) - lead; };
        if (wm) {
          uint32_t at = S.base_above + atomicAdd(&S.ctr_win, uint32_t(__popc(wm)));
          for (; wm; wm &= wm - 1u, ++at) {
            const int j = __ffs(wm) - 1;
            if (at < uint32_t(k)) {  // always true: counts match the histogram's
              out[at] = window_of(j);
              if (outv) outv[at] = stage_score(slot, c0, j);
            }
          }
        }
        if (cm) {
          uint32_t c = S.base_cand + atomicAdd(&S.ctr_cand, uint32_t(__popc(cm)));
          for (; cm; cm &= cm - 1u, ++c) {
            const int j = __ffs(cm) - 1;
            if (c < cand_cap) {  // always true: m fits the buffer on this path
              dsmem_st_u32(rv + 4u * c, __float_as_uint(stage_score(slot, c0, j)));
              dsmem_st_u32(rj + 4u * c, uint32_t(window_of(j)));
            }
          }
        }
      };
      if (rank == 0 && !cand_in_list)
        global_pass(visit);  // rank 0's ring receives the candidates
      else
        stream_pass(false, collect_stage);
      report_timeout();
    }
    csync();  // every candidate has landed in rank 0's buffer
    if (rank != 0) return;

    // ------------------------------------------------------------ refine (rank 0)
    const uint32_t need = uint32_t(k) - cr.above;
    const uint32_t mm = cr.m < cand_cap ? cr.m : cand_cap;
    if ((mm <= uint32_t(RANK_REFINE_MAX) && !(p.flags & FLAG_RADIX_REFINE)) || det) {
      // (deterministic mode ranks every candidate set: ties by smallest index)
      // rank of candidate i = number of candidates ordered before it by (value desc, index asc)
      static_assert(CAP % 4 == 0, "the candidate arrays start 16-byte aligned");
      for (uint32_t i = tid; i < mm; i += T) {
        const float v = cand_v[i];
        const int32_t j = cand_j[i];
        uint32_t r = 0;
        uint32_t q = 0;
        for (; q + 4 <= mm; q += 4) {  // four candidates per pair of 16-byte loads
          const float4 w = *reinterpret_cast<const float4*>(cand_v + q);
          const int4 jj = *reinterpret_cast<const int4*>(cand_j + q);
          r += uint32_t((w.x > v) || (w.x == v && jj.x < j)) + uint32_t((w.y > v) || (w.y == v && jj.y < j)) +
               uint32_t((w.z > v) || (w.z == v && jj.z < j)) + uint32_t((w.w > v) || (w.w == v && jj.w < j));
        }
        for (; q < mm; ++q) {
          const float w = cand_v[q];
          const int32_t jj = cand_j[q];
          r += (w > v) || (w == v && jj < j);
        }
        if (r < need && cr.above + r < uint32_t(k)) {
          out[cr.above + r] = j;
          if (outv) outv[cr.above + r] = v;
        }
      }
    } else {
      // The candidates' smallest and largest order key: the digits they share are fixed before
      // the first digit pass (a crossing bin is narrow, its keys usually share one or two bytes),
      // and equal keys are all ties at once.
      uint32_t kmin = 0xffffffffu, kmax = 0u;
      for (uint32_t i = tid; i < mm; i += T) {
        const uint32_t key = order_key(cand_v[i]);
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
      kmin = __reduce_min_sync(FULL_MASK, kmin);
      kmax = __reduce_max_sync(FULL_MASK, kmax);
      if (tid == 0) {
        S.kmin_loc = 0xffffffffu;
        S.kmax_loc = 0u;
      }
      __syncthreads();
      if (lane == 0) {
        atomicMin(&S.kmin_loc, kmin);
        atomicMax(&S.kmax_loc, kmax);
      }
      __syncthreads();
      kmin = S.kmin_loc;
      kmax = S.kmax_loc;
      const int dfix = kmin == kmax ? 4 : __clz(kmin ^ kmax) / 8;  // whole shared bytes
      uint32_t prefix = dfix >= 4 ? kmin : (dfix > 0 ? kmin & (0xffffffffu << (32 - 8 * dfix)) : 0u);
      uint32_t pmask = dfix >= 4 ? 0xffffffffu : (dfix > 0 ? 0xffffffffu << (32 - 8 * dfix) : 0u);
      uint32_t rneed = need;
      bool ge = false;
      for (int pass = dfix; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += T) digit_hist(S, 0)[i] = 0;
        __syncthreads();
        for (uint32_t b0 = 0; b0 < mm; b0 += T) {
          const uint32_t i = b0 + tid;
          const bool in = i < mm;
          const uint32_t key = in ? order_key(cand_v[i]) : 0u;
          const bool pr = in && (key & pmask) == prefix;
          if (pr) atomicAdd(&digit_hist(S, 0)[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        // the digit where rneed is reached, from this CTA's own counts (plain shared loads)
        const DigitCross dc = digit_scan<T>(S, digit_hist(S, 0), digit_hist(S, 0), rneed);
        prefix |= dc.digit << shift;
        pmask |= 0xFFu << shift;
        rneed -= dc.above;
        __syncthreads();
        if (dc.cnt == rneed) {
          ge = true;
          break;
        }
      }
      const uint32_t nties = ge ? 0u : rneed;
      const uint32_t win_base = cr.above, tie_base = cr.above + (need - nties);
      // emission with no warp collective: each thread counts its winners and ties, takes their
      // slots with one shared atomic per kind, then writes them
      uint32_t nw = 0, nt = 0;
      for (uint32_t i = tid; i < mm; i += T) {
        const uint32_t key = order_key(cand_v[i]);
        nw += (ge ? (key & pmask) >= prefix : key > prefix) ? 1u : 0u;
        nt += (!ge && key == prefix) ? 1u : 0u;
      }
      uint32_t ws = nw ? atomicAdd(&S.ctr_rwin, nw) : 0u;
      uint32_t ts = nt ? atomicAdd(&S.ctr_rtie, nt) : 0u;
      if (nw | nt)
        for (uint32_t i = tid; i < mm; i += T) {
          const uint32_t key = order_key(cand_v[i]);
          if (ge ? (key & pmask) >= prefix : key > prefix) {
            if (win_base + ws < tie_base) {
              out[win_base + ws] = cand_j[i];
              if (outv) outv[win_base + ws] = cand_v[i];
            }
            ++ws;
          } else if (!ge && key == prefix) {
            if (ts < nties) {
              out[tie_base + ts] = cand_j[i];
              if (outv) outv[tie_base + ts] = cand_v[i];
            }
            ++ts;
          }
        }
    }
    __syncthreads();
    const bool failed = S.err || S.tout;
    if (failed)
      for (int i = tid; i < k; i += T) out[i] = -2;
    else if (EXT && (p.flags & FLAG_SORTED))
      sort_output();
    if (stats) {
      stats[0] = failed ? PATH_DEVICE_ERROR : PATH_REFINE;
      stats[1] = int32_t(cr.m);
      stats[2] = rounds;
      stats[3] = int32_t(cr.above);
    }
    return;
  }

  // ---------------------------------------------------------------- re-list
  // The crossing bin holds more candidates than the buffer and some CTA's first-pass list
  // overflowed: every CTA lists only the scores of the crossing bin and above (one list per
  // CTA) -- a CTA whose first-pass list is complete filters it in place, the others read their
  // share once more.  When every such list fits, the selection below runs over the lists;
  // otherwise it reads the row.  Rows whose crossing bin and above cannot fit in the cluster's
  // lists (tie-heavy rows) go to the row-wide selection at once.
  if (path == PATH_RESCUE_OVERFLOW && cr.total >= uint32_t(k) && !(p.flags & FLAG_STREAM_RESCUE) &&
      uint64_t(cr.above) + cr.m <= uint64_t(cs) * LCAP) {
    if (warp == 0) {
      const float t = cr.bin > 0 ? floor_value(cr.bin, gmin, sc) : -INFINITY;
      if (lane == 0) S.vthr = t;
    }
    __syncthreads();
    const float tb = fmaxf(S.vthr, cthr);  // scores >= tb: the crossing bin's members and above
    if (rounds == 1 && listed) {
      // Compact the first-pass list (walk order, segments in turn) to the entries >= tb.  An
      // entry is written below the walk index of every entry not read yet, so one barrier per
      // round between the reads and the writes keeps unread entries intact.
      uint32_t pre[NW + 1];
      pre[0] = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) pre[w + 1] = pre[w] + S.list_n[w];
      for (uint32_t b0 = 0; b0 < pre[NW]; b0 += T) {
        const uint32_t i = b0 + tid;
        const bool in = i < pre[NW];
        uint32_t at = i;
#pragma unroll
        for (int w = 1; w < NW; ++w)
          if (i >= pre[w]) at = uint32_t(w * LSEG) + (i - pre[w]);
        const float v = in ? list_val(at) : 0.f;
        const uint32_t key = in ? list_keyat(at) : 0u;
        const bool hit = in && v >= tb;
        __syncthreads();
        const uint32_t slot = warp_alloc_local(&S.relist_n, hit);
        if (hit) list_put(slot, v, key);
      }
      __syncthreads();
    } else {
      stream_pass(false, [&](uint32_t slot, int32_t c0) {
        each_lane(slot, c0, [&](float e, int32_t g, bool valid, int l) {
          const bool hit = valid && e >= tb;
          if (__any_sync(FULL_MASK, hit)) {
            const uint32_t at = warp_alloc_local(&S.relist_n, hit);
            if (hit && at < uint32_t(LCAP)) list_put(at, e, list_key(g, l));
          }
        });
      });
      rounds += 10;  // diagnostics: the share was read again
    }
    if (tid == 0) {
      const bool fits = S.relist_n <= uint32_t(LCAP) && (!L16 || nstages <= LIST_MAX_STAGES);
#pragma unroll
      for (int w = 0; w < NW; ++w) S.list_n[w] = 0;
      S.list_n[0] = fits ? S.relist_n : 0u;  // one contiguous list
      if (!fits)
        for (uint32_t c = 0; c < cs; ++c) dsmem_red_add(dsmem_map(smem_u32(&S.relist_bad), c), 1u);
    }
    csync();
    report_timeout();
    if (S.relist_bad == 0) path = PATH_REFINE_RELIST;
  }

  // ---------------------------------------------------------------- rescue: cluster radix select
  // Exact selection over the 32-bit order-preserving keys, one 8-bit digit per pass from the
  // top.  Each pass counts the digits of the keys that still match the chosen prefix, pushes
  // the counts (and the smallest / largest matching key) into every CTA, and fixes one digit
  // of tau's key.  It stops early when the digits above the chosen one already account for
  // exactly the keys still needed, or when every matching key is the same (tie-heavy rows).
  // Positions outside the window are masked by position.
  // After a valid histogram the selection is seeded with it: only the counted scores of the
  // crossing bin take part, k - above of them are needed, and every score of a higher bin is a
  // winner.  When every CTA's list held its counted scores, the passes read the lists instead
  // of the row.
  const bool from_lists = path == PATH_REFINE_CLUSTER || path == PATH_REFINE_RELIST;
  const bool seeded = from_lists || (path == PATH_RESCUE_OVERFLOW && cr.total >= uint32_t(k));
  const int bstar = cr.bin;
  uint32_t* dloc = S.hist;  // this CTA's digit counts
  auto dtot = [&](int buf) -> uint32_t* { return S.tot + 256 * buf; };
  auto kslot = [&](int buf, int which) -> uint32_t* { return S.tot + 512 + 2 * buf + which; };
  for (int i = tid; i < 512; i += T) S.tot[i] = 0;
  if (tid == 0) {
    *kslot(0, 0) = *kslot(1, 0) = 0xffffffffu;
    *kslot(0, 1) = *kslot(1, 1) = 0u;
  }
  __syncthreads();
  csync();  // every CTA's pushed totals start from zero
  bool primed = rounds == 0;  // the head primed the ring for a row without a first pass
  // Bin class of a score for the seeded selection: 1 above the crossing bin, 0 a member of it,
  // -1 below it (or not counted).  Unseeded, every score is a member.
  uint32_t klo = 0, khi = KEY_POS_INF;
  // Seeded, every member's key lies in [klo, khi] (the crossing bin's value range, and >= cthr):
  // the digits that klo and khi share are fixed before the first pass (at least one pass runs).
  uint32_t tau_prefix = 0, tau_mask = 0;
  int tau_shift = 24;
  if (seeded) {
    if (warp == 0) {
      const float lo = bstar > 0 ? floor_value(bstar, gmin, sc) : -INFINITY;
      const float hi = bstar < NB - 1 ? floor_value(bstar + 1, gmin, sc) : INFINITY;
      if (lane == 0) {
        S.klo = order_key(fmaxf(lo, cthr));
        S.khi = bstar < NB - 1 ? order_key(hi) - 1u : KEY_POS_INF;
      }
    }
    __syncthreads();
    klo = S.klo;
    khi = S.khi;
    const int dfix = klo <= khi ? min(__clz(klo ^ khi) / 8, 3) : 0;
    if (dfix > 0) {
      tau_mask = 0xffffffffu << (32 - 8 * dfix);
      tau_prefix = klo & tau_mask;
      tau_shift = 24 - 8 * dfix;
    }
  }
  // Class of a score by its order key, for the seeded selection: 1 above the crossing bin, 0 a
  // member of it (a counted score of the bin: key in [klo, khi]), -1 below it, uncounted or NaN
  // (whose keys lie beyond +inf's or below -inf's).  Unseeded, every score is a member.
  auto key_class = [&](uint32_t key) -> int {
    if (!seeded) return 0;
    if (key > KEY_POS_INF) return -1;
    return key > khi ? 1 : (key >= klo ? 0 : -1);
  };
  // One cluster radix selection: the `need` largest keys among the scores that sel(e, j, key)
  // admits (it also computes the key), one 8-bit digit per pass from bit shift0 down, below the
  // fixed key bits (prefix0 under pmask0).  The result is the selected keys' boundary: with ge
  // the keys whose masked value is >= prefix are exactly the selected ones; without ge the keys
  // above prefix are, plus `need` of the keys equal to prefix (pmask is then all ones).
  // my_above / my_at: this CTA's admitted scores above / at the boundary.
  struct Sel {
    uint32_t prefix, pmask, need, my_above, my_at;
    bool ge;
    bool first_eq;  // the first pass found every admitted key equal (all of them are tau)
  };
  int rpass = 0;  // digit-total buffers alternate over the passes of every selection
  // record: the first pass also keeps the window indices of up to REC_CAP admitted scores of this
  // CTA (in the idle list area), so that a tie class found in that pass needs no emission read.
  int32_t* const rec = reinterpret_cast<int32_t*>(&S.list_v[0]);  // the whole list area: REC_CAP int32
  auto radix_select = [&](auto&& sel, uint32_t need0, uint32_t prefix0, uint32_t pmask0, int shift0,
                          bool record) -> Sel {
    Sel r{prefix0, pmask0, need0, 0u, 0u, false, false};
    if (tid == 0) S.rec_n = 0;
    for (int shift = shift0; shift >= 0; shift -= 8) {
      const int buf = rpass++ & 1;
      for (int i = tid; i < 256; i += T) dloc[i] = 0;
      if (tid == 0) {
        S.kmin_loc = 0xffffffffu;
        S.kmax_loc = 0u;
      }
      __syncthreads();
      uint32_t tmin = 0xffffffffu, tmax = 0u;
      // Count the digits of a thread's batch of N scores (bit j of vm: score j is in the
      // window).  Warp-collective.  A warp whose admitted keys all share one digit adds them
      // with one atomic (tie-heavy and narrow rows); otherwise one atomic per distinct digit per
      // score slot.
      auto digit_batch = [&](auto n_c, const auto& e, const auto& jw, uint32_t vm) {  // arrays of N, by reference
        constexpr int N = decltype(n_c)::value;
        uint32_t keys[N];
        uint32_t pm = 0, dmin = 0xffffffffu, dmax = 0u;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          uint32_t key = 0;
          const bool ok = ((vm >> j) & 1u) && sel(e[j], jw[j], key) && (key & r.pmask) == r.prefix;
          keys[j] = key;
          if (ok) {
            pm |= 1u << j;
            tmin = min(tmin, key);
            tmax = max(tmax, key);
            const uint32_t d = (key >> shift) & 255u;
            dmin = min(dmin, d);
            dmax = max(dmax, d);
          }
        }
        if (record && shift == shift0 && S.rec_n < REC_CAP) {  // warp-uniform
          const uint32_t nm = __popc(pm);
          const unsigned lt = lanemask_lt();
          uint32_t excl = 0, wtot = 0;
#pragma unroll
          for (int b = 0; (1 << b) <= N; ++b) {
            const unsigned m = __ballot_sync(FULL_MASK, (nm >> b) & 1u);
            excl += uint32_t(__popc(m & lt)) << b;
            wtot += uint32_t(__popc(m)) << b;
          }
          uint32_t base = 0;
          if (lane == 0 && wtot) base = atomicAdd(&S.rec_n, wtot);
          uint32_t at = __shfl_sync(FULL_MASK, base, 0) + excl;
#pragma unroll
          for (int j = 0; j < N; ++j)
            if ((pm >> j) & 1u) {
              if (at < REC_CAP) rec[at] = jw[j];
              ++at;
            }
        }
        dmin = __reduce_min_sync(FULL_MASK, dmin);
        dmax = __reduce_max_sync(FULL_MASK, dmax);
        if (dmin == dmax) {
          const uint32_t c = __reduce_add_sync(FULL_MASK, uint32_t(__popc(pm)));
          if (lane == 0) atomicAdd(&dloc[dmin], c);
        } else if (dmin < dmax) {  // plain atomics: the hardware merges lanes on one digit
#pragma unroll
          for (int j = 0; j < N; ++j)
            if ((pm >> j) & 1u) atomicAdd(&dloc[(keys[j] >> shift) & 255u], 1u);
        }
      };
      if (from_lists) {
        each_listed([&](float v, int32_t j, bool in) {
          const float e[1] = {v};
          const int32_t jj[1] = {j};
          digit_batch(IntC<1>{}, e, jj, in ? 1u : 0u);
        });
      } else {
        stream_pass(primed, [&](uint32_t slot, int32_t c0) {
          float e[4 * VPS];
          int32_t jw[4 * VPS];
          uint32_t vm = 0xffffffffu;
          if (c0 > 0 && c0 + STAGE_VEC <= ffull) {  // an interior stage: every lane is in the window
#pragma unroll
            for (int i = 0; i < VPS; ++i) {
              const float4 v = ring[slot][i * T + tid];
#pragma unroll
              for (int l = 0; l < 4; ++l) {
                e[4 * i + l] = f4_get(v, l);
                jw[4 * i + l] = 4 * (c0 + i * T + tid) + l - lead;
              }
            }
          } else {
            vm = 0;
#pragma unroll
            for (int i = 0; i < VPS; ++i) {
              int32_t g;
              float4 v;
              vm |= stage_vec(slot, c0, i, g, v) << (4 * i);
#pragma unroll
              for (int l = 0; l < 4; ++l) {
                e[4 * i + l] = f4_get(v, l);
                jw[4 * i + l] = 4 * g + l - lead;
              }
            }
          }
          digit_batch(IntC<4 * VPS>{}, e, jw, vm);
        });
      }
      primed = false;
      tmin = __reduce_min_sync(FULL_MASK, tmin);
      tmax = __reduce_max_sync(FULL_MASK, tmax);
      if (lane == 0) {
        atomicMin(&S.kmin_loc, tmin);
        atomicMax(&S.kmax_loc, tmax);
      }
      __syncthreads();
      for (int d = tid; d < 256; d += T) {
        const uint32_t v = dloc[d];
        if (v) {
          const uint32_t local = smem_u32(&dtot(buf)[d]);
          for (uint32_t c = 0; c < cs; ++c) dsmem_red_add(dsmem_map(local, c), v);
        }
      }
      if (tid == 0)
        for (uint32_t c = 0; c < cs; ++c) {
          dsmem_red_min(dsmem_map(smem_u32(kslot(buf, 0)), c), S.kmin_loc);
          dsmem_red_max(dsmem_map(smem_u32(kslot(buf, 1)), c), S.kmax_loc);
        }
      csync();
      report_timeout();
      const DigitCross dc = digit_scan<T>(S, dtot(buf), dloc, r.need);
      const uint32_t kmin_all = *kslot(buf, 0), kmax_all = *kslot(buf, 1);
      __syncthreads();  // every thread has read this pass's totals: reset them for two passes on
      for (int i = tid; i < 256; i += T) dtot(buf)[i] = 0;
      if (tid == 0) {
        *kslot(buf, 0) = 0xffffffffu;
        *kslot(buf, 1) = 0u;
      }
      if (kmin_all == kmax_all) {  // every admitted key with this prefix is the same
        r.prefix = kmin_all;
        r.pmask = 0xffffffffu;
        r.my_at = dc.my_all;
        r.first_eq = shift == shift0;
        break;
      }
      r.prefix |= dc.digit << shift;
      r.pmask |= 0xFFu << shift;
      r.need -= dc.above;
      r.my_above += dc.my_above;
      r.my_at = dc.my_at;
      if (dc.cnt == r.need) {  // the keys with this prefix are exactly the remaining ones
        r.ge = true;
        r.my_above += dc.my_at;
        r.my_at = 0;
        break;
      }
    }
    return r;
  };
  // One value above the floor: the first pass found every score >= thr equal (its smallest and
  // largest keys agree cluster-wide), so the crossing bin's members are one tie class, tau is
  // that value, nothing lies above it, and any k of them are the selection.  When the lists hold
  // at least k of them, the tie slots come from the lists: no digit pass, no second read.
  const bool one_value = seeded && !from_lists && !bmax_row && !det && rounds == 1 && S.hk_min == S.hk_max &&
                         cr.above == 0 && S.hlisted >= uint32_t(k);
  if (one_value) {
    uint32_t lpre[NW + 1];  // listed entries before each warp's segment
    lpre[0] = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) lpre[w + 1] = lpre[w] + min(S.list_n[w], uint32_t(LSEG));
    const uint32_t my_eq = lpre[NW];
    if (tid == 32) S.base_cand = my_eq ? dsmem_atom_add(dsmem_map(smem_u32(&S.rc_tie), 0), my_eq) : 0u;
    __syncthreads();
    const uint32_t tbase = S.base_cand;
    const uint32_t my_ties = tbase < uint32_t(k) ? min(my_eq, uint32_t(k) - tbase) : 0u;
    for (uint32_t i = tid; i < my_ties; i += T) {
      uint32_t at = i;  // segment w holds entries lpre[w] ..: static indices only
#pragma unroll
      for (int q = 1; q < NW; ++q)
        if (i >= lpre[q]) at = uint32_t(q * LSEG) + (i - lpre[q]);
      out[tbase + i] = list_window(at);
      if (outv) outv[tbase + i] = list_val(at);
    }
  } else {
    // tau: the k - above largest order keys among the members
    const Sel t = radix_select([&](float e, int32_t, uint32_t& key) {
      key = order_key(e);
      return key_class(key) == 0;
    }, seeded ? uint32_t(k) - cr.above : uint32_t(k), tau_prefix, tau_mask, tau_shift, !from_lists);
    const uint32_t prefix = t.prefix, pmask = t.pmask;
    const bool ge = t.ge;
    const uint32_t my_win = (seeded ? cr.my_above : 0u) + t.my_above;  // this CTA's scores above tau
    const uint32_t nties = ge ? 0u : t.need;                           // tie slots
    // Deterministic mode: the tie slots go to the ties with the smallest window indices, the
    // nties largest keys ~j among the scores equal to tau.  Keys of indices below 2^(8D) share
    // their top 32 - 8D bits (all ones), so only D digit passes are needed.
    bool by_index = false;
    Sel ix{};
    if (det && nties > 0) {
      by_index = true;
      const int digits = (32 - __clz(int(nv - 1u)) + 7) / 8;
      const uint32_t fixed = digits < 4 ? (0xffffffffu << (8 * digits)) : 0u;
      ix = radix_select([&](float e, int32_t jw, uint32_t& key) {
        key = ~uint32_t(jw);
        const uint32_t kv = order_key(e);
        return key_class(kv) == 0 && kv == prefix;
      }, nties, fixed, fixed, 8 * (digits - 1), false);
    }
    auto index_selected = [&](int32_t jw) -> bool {
      const uint32_t key = ~uint32_t(jw);
      return ix.ge ? (key & ix.pmask) >= ix.prefix : key >= ix.prefix;
    };
    // this CTA's tie candidates for the slots: all its ties, or its index-selected ties
    const uint32_t my_eq = by_index ? ix.my_above + (ix.ge ? 0u : ix.my_at) : t.my_at;
    // Emission: rank 0 hands this CTA a block of winner slots and a block of tie slots.
    const uint32_t tie_base = uint32_t(k) - nties;
    if (tid == 0) S.base_above = my_win ? dsmem_atom_add(dsmem_map(smem_u32(&S.rc_win), 0), my_win) : 0u;
    if (tid == 32) S.base_cand = my_eq ? dsmem_atom_add(dsmem_map(smem_u32(&S.rc_tie), 0), my_eq) : 0u;
    __syncthreads();
    const uint32_t wbase = S.base_above, tbase = S.base_cand;
    // ties this CTA writes: its share of the nties slots, in the order the slots were handed out
    const uint32_t my_ties = tbase < nties ? (my_eq < nties - tbase ? my_eq : nties - tbase) : 0u;
    auto emit = [&](float e, int32_t jw, bool valid) {  // warp-collective
      const uint32_t key = order_key(e);
      const int bc = valid ? key_class(key) : -1;
      const bool win = bc == 1 || (bc == 0 && (ge ? (key & pmask) >= prefix : key > prefix));
      const bool tie = bc == 0 && !ge && key == prefix && (!by_index || index_selected(jw));
      const uint32_t ws = warp_alloc_local(&S.ctr_win, win);
      if (win && wbase + ws < tie_base) {
        out[wbase + ws] = jw;
        if (outv) outv[wbase + ws] = e;
      }
      const uint32_t ts = warp_alloc_local(&S.ctr_cand, tie);
      if (tie && tbase + ts < nties) {
        out[tie_base + tbase + ts] = jw;
        if (outv) outv[tie_base + tbase + ts] = e;
      }
    };
    // A tie class found by the first digit pass, with nothing above it in this CTA: the tie slots
    // come from the indices that pass recorded, without another read of the share.
    const uint32_t recorded = min(S.rec_n, REC_CAP);
    if (t.first_eq && !from_lists && !by_index && my_win == 0 && my_ties > 0 && my_ties <= recorded) {
      for (uint32_t i = tid; i < my_ties; i += T) {
        const int32_t jw = rec[i];
        out[tie_base + tbase + i] = jw;
        if (outv) outv[tie_base + tbase + i] = __ldg(rowp + a + uint32_t(jw));
      }
    } else if (my_win > 0 || my_ties > 0) {
      if (from_lists) {
        each_listed([&](float e, int32_t jw, bool in) { emit(e, jw, in); });
      } else {
        static_assert(4 * VPS < 16, "a thread's slot count per stage fits in 4 bits");
        stream_pass(false, [&](uint32_t slot, int32_t c0) {
          // stop visiting once this CTA's slots are all handed out (the counters only grow, and a
          // warp reads them together; the remaining stages still land and are waited for)
          if (S.ctr_win >= my_win && S.ctr_cand >= my_ties) return;
          // Each thread marks its winners and ties of the stage (bit 4i + l), the warp takes its
          // slots of each kind with one atomic, and each thread writes its own in turn.
          uint32_t wm = 0, tm = 0;
          each_lane(slot, c0, [&](float e, int32_t g, bool valid, int l) {
            const uint32_t key = order_key(e);
            const int bc = valid ? key_class(key) : -1;
            const bool win = bc == 1 || (bc == 0 && (ge ? (key & pmask) >= prefix : key > prefix));
            const bool tie = bc == 0 && !ge && key == prefix && (!by_index || index_selected(4 * g + l - lead));
            const int j = 4 * ((g - c0) / T) + l;
            wm |= uint32_t(win) << j;
            tm |= uint32_t(tie) << j;
          });
          uint32_t ws = warp_alloc_n(&S.ctr_win, __popc(wm));
          uint32_t ts = warp_alloc_n(&S.ctr_cand, __popc(tm));
          auto put = [&](int j, uint32_t at) {
            out[at] = 4 * (c0 + (j >> 2) * T + tid) + (j & 3) - lead;
            if (outv) outv[at] = stage_score(slot, c0, j);
          };
          for (uint32_t rest = wm; rest; rest &= rest - 1, ++ws)
            if (wbase + ws < tie_base) put(__ffs(rest) - 1, wbase + ws);
          for (uint32_t rest = tm; rest; rest &= rest - 1, ++ts)
            if (tbase + ts < nties) put(__ffs(rest) - 1, tie_base + tbase + ts);
        });
      }
    }
  }
  report_timeout();
  csync();  // rank 0's counters stay alive until every CTA is done with them
  if (rank == 0) {
    const bool failed = S.err || S.tout;
    if (failed)
      for (int i = tid; i < k; i += T) out[i] = -2;
    else if (EXT && (p.flags & FLAG_SORTED))
      sort_output();
    if (stats) {
      stats[0] = failed ? PATH_DEVICE_ERROR : path;
      stats[1] = int32_t(cr.m);
      stats[2] = rounds;
      stats[3] = seeded ? int32_t(cr.above) : 0;
    }
  }
}

}  // namespace gvr
