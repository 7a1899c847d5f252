// gvr_short.cuh -- GVR top-K for short rows (row stride <= 16384 scores): one CTA per row, the
// whole window resident in shared memory.
//
// The cluster kernel (gvr_kernel.cuh) streams a row through a small shared-memory ring so that
// rows of any length work; for a short row that costs a latency chain per ring stage, cluster
// exchanges, and a long stretch of code that every CTA runs once (with few rows on the GPU its
// instructions come in cold).  Here one CTA of 1024 threads takes a whole row: thread 0 stages the
// window in shared memory with a few bulk copies (TMA) completing on one mbarrier, and while they
// are in flight every thread loads its block64 samples ("GVR K=2048 reg_clus with block64
// sampling and parallel rescue", TensorRT-LLM PR #20998, "What changes") and the CTA reduces them
// to the bracket [GMIN, GMAX] and the sampled floor t.  Then, over the resident window:
//
//   Verify  the scores >= t are counted in NB value bins (shared memory) and a suffix scan finds
//           the bin that crosses the K-th largest score ("Why the GLM row overflows");
//   Refine  the winners of the bins above it are written, the crossing bin's members gathered
//           and the k - above largest of them picked exactly (rank counting, or a radix select
//           on their order keys);
//   Rescue  an invalid bracket, fewer than k scores at or above t, or a crossing bin larger than
//           the gather buffer take an exact radix select over the order keys of the window
//           (4 digit passes at most, early exits).
//
// Every pass is a short rolled loop over shared memory in which a vector with no score at or
// above the floor costs one compare of its largest lane; 32 warps per row keep enough
// independent work in flight to hide the latency of each thread's short chain.  No cluster, no
// ring, no distributed shared memory.
#pragma once

#include "gvr_kernel.cuh"

namespace gvr {

constexpr int SHORT_THREADS = 1024;
constexpr int SHORT_MAX = 16384;   // row stride (scores) whose window the kernel holds
constexpr int SHORT_CAND = 2048;   // crossing-bin members it gathers at most
constexpr int SHORT_LIST = 4096;   // scores at or above the floor it lists at most
constexpr uint32_t SHORT_COPY_VEC = 256;     // float4 per bulk copy (4 KB)
constexpr int PATH_SHORT_KERNEL = 10;        // row_stats: selected by the short-row kernel
constexpr int PATH_SHORT_KERNEL_RADIX = 11;  // row_stats: ... by its radix select over the row

struct ShortParams {
  const float* logits;
  int64_t row_stride;
  const int32_t* kv_lens;     // decode
  const int32_t* row_starts;  // prefill
  const int32_t* row_ends;    // prefill
  int32_t* indices;
  float* values;              // nullable
  int32_t* row_stats;         // nullable, [rows][4]
  int32_t next_n;
  int32_t compress_ratio;
  int32_t k;
  int32_t mode;
  int32_t flags;              // FLAG_FORCE_RESCUE, FLAG_DIAG_FAIL_ROW0 or 0
};

struct alignas(16) ShortSmem {
  uint32_t hist[NB + 4];   // samples' histogram, then the scores' histogram, then digit counts
  uint16_t list[SHORT_LIST];  // positions (in the staged vectors) of the scores at or above the floor
  uint16_t cand[SHORT_CAND];  // positions of the crossing bin's members
  uint64_t bar;            // the window's bulk copies
  uint32_t wsum[32];
  float wmin[32], wmax[32];
  int32_t sel;
  uint32_t sel_before, sel_at;
  uint32_t kmin_loc, kmax_loc;
  uint32_t ctr_win, ctr_cand, ctr_tie, list_n;
  uint32_t tout;
};
static_assert(offsetof(ShortSmem, hist) % 16 == 0, "histograms are read as 16-byte vectors");
static_assert(offsetof(ShortSmem, bar) % 8 == 0, "mbarrier alignment");

// The window follows the header: vector g holds window positions 4g - lead .. 4g + 3 - lead of
// a window read from the 16-byte boundary at or below its start (lead = start mod 4); at most
// stride / 4 full vectors and the partial last one.
constexpr size_t SHORT_HDR = (sizeof(ShortSmem) + 15) / 16 * 16;
__host__ __device__ constexpr size_t short_smem_bytes(int64_t row_stride) {
  return SHORT_HDR + 16 * size_t(row_stride / 4 + 1);
}

// One count per thread, in descending order of what they count (thread 0 first): the thread
// where the running count reaches `want` (-1 when the total stays below it), with the count
// before it and its own.  Block-collective over SHORT_THREADS threads.  Each shared word is
// written only after a barrier that every reader of its previous value has passed, so calls may
// follow one another with no barrier between them.  Two barriers.
struct ShortCross {
  int32_t t;
  uint32_t before, at;
};
__device__ __forceinline__ ShortCross short_cross(ShortSmem& S, uint32_t c, uint32_t want) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  static_assert(SHORT_THREADS == 1024, "each lane reads one warp's sum");
  uint32_t it = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(FULL_MASK, it, o);
    if (lane >= o) it += x;
  }
  if (lane == 31) S.wsum[warp] = it;
  __syncthreads();
  // every warp scans the 32 warp sums itself (no second barrier)
  const uint32_t w = S.wsum[lane];
  uint32_t iw = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(FULL_MASK, iw, o);
    if (lane >= o) iw += x;
  }
  const uint32_t before = __shfl_sync(FULL_MASK, iw - w, warp) + it - c;
  const uint32_t total = __shfl_sync(FULL_MASK, iw, 31);
  if (before < want && before + c >= want) {  // one thread at most: the running count crosses once
    S.sel = tid;
    S.sel_before = before;
    S.sel_at = c;
  }
  __syncthreads();
  if (total < want) return ShortCross{-1, 0u, 0u};
  return ShortCross{S.sel, S.sel_before, S.sel_at};
}

// Each thread's first slot of n from a shared counter: an exclusive prefix over the warp and one
// atomic per warp.  Warp-collective.
__device__ __forceinline__ uint32_t warp_slots(uint32_t* c, uint32_t n) {
  const int lane = threadIdx.x & 31;
  uint32_t i = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(FULL_MASK, i, o);
    if (lane >= o) i += x;
  }
  uint32_t b = 0;
  if (lane == 31 && i) b = atomicAdd(c, i);
  return __shfl_sync(FULL_MASK, b, 31) + i - n;
}

// Each thread's first slots of two kinds (na of the first, nb of the second) from two shared
// counters: an exclusive prefix over the warp and one atomic per counter and warp.  Warp-collective.
__device__ __forceinline__ void warp_slots2(uint32_t* ca, uint32_t* cb, uint32_t na, uint32_t nb, uint32_t& sa,
                                            uint32_t& sb) {
  const int lane = threadIdx.x & 31;
  uint32_t ia = na, ib = nb;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(FULL_MASK, ia, o), y = __shfl_up_sync(FULL_MASK, ib, o);
    if (lane >= o) {
      ia += x;
      ib += y;
    }
  }
  uint32_t ba = 0, bb = 0;
  if (lane == 31) {
    if (ia) ba = atomicAdd(ca, ia);
    if (ib) bb = atomicAdd(cb, ib);
  }
  sa = __shfl_sync(FULL_MASK, ba, 31) + ia - na;
  sb = __shfl_sync(FULL_MASK, bb, 31) + ib - nb;
}

// The window's scores that may reach the floor: vector g with the lanes before the window start
// (vector 0 only) set to -inf; the partial last vector's lanes past the window are NaN already.
__device__ __forceinline__ float4 short_masked(float4 x, uint32_t g, uint32_t lead) {
  if (g == 0 && lead) {
    x.x = -INFINITY;
    if (lead > 1) x.y = -INFINITY;
    if (lead > 2) x.z = -INFINITY;
  }
  return x;
}

__global__ void __launch_bounds__(SHORT_THREADS, 2) gvr_short_kernel(const ShortParams p) {
  constexpr int T = SHORT_THREADS;
  constexpr int NW = T / 32;
  constexpr int KPT = MAX_SAMPLES / T;  // samples per thread at most
  extern __shared__ __align__(16) unsigned char short_smem[];
  ShortSmem& S = *reinterpret_cast<ShortSmem*>(short_smem);
  float4* const rv = reinterpret_cast<float4*>(short_smem + SHORT_HDR);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t row = blockIdx.x;
  const int32_t k = p.k;
  const float qnan = __int_as_float(0x7fffffff);

  // ---------------------------------------------------------------- row geometry
  const uint32_t stride = uint32_t(p.row_stride);
  uint32_t a = 0, nv = 0;
  if (p.mode == MODE_DECODE) {
    const uint32_t nn = uint32_t(p.next_n);
    const uint32_t req = row / nn;
    const int32_t kv = __ldg(p.kv_lens + req);
    if (kv >= p.next_n) nv = (uint32_t(kv) - nn + (row - req * nn) + 1u) / uint32_t(p.compress_ratio);
    nv = nv < stride ? nv : stride;
  } else {
    const int32_t ks = __ldg(p.row_starts + row);
    const int32_t ke = __ldg(p.row_ends + row);
    const uint32_t s = ks > 0 ? uint32_t(ks) : 0u;
    const uint32_t e = ke > 0 ? (uint32_t(ke) < stride ? uint32_t(ke) : stride) : 0u;
    a = s < stride ? s : stride;
    nv = e > a ? e - a : 0u;
  }
  const float* rowp = p.logits + int64_t(row) * p.row_stride;
  int32_t* out = p.indices + int64_t(row) * k;
  float* outv = p.values ? p.values + int64_t(row) * k : nullptr;
  int32_t* stats = (p.row_stats && tid == 0) ? p.row_stats + 4 * int64_t(row) : nullptr;
  if (nv <= uint32_t(k)) {  // identity and -1 pad
    for (int i = tid; i < k; i += T) {
      out[i] = uint32_t(i) < nv ? i : -1;
      if (outv) outv[i] = uint32_t(i) < nv ? rowp[a + i] : -FLT_MAX;
    }
    if (stats) {
      stats[0] = PATH_SHORT;
      stats[1] = stats[2] = stats[3] = 0;
    }
    return;
  }

  // ---------------------------------------------------------------- the window into shared memory
  // Full vectors by bulk copies from the aligned start (a window never ends past its row, so
  // neither do they); the partial last vector as scalars, never past the window.
  const uint32_t lead = a & 3u;
  const float* base = rowp + (a - lead);
  const uint32_t span = lead + nv;
  const uint32_t ffull = span >> 2, tailn = span & 3u;
  const uint32_t nvec = ffull + (tailn ? 1u : 0u);
  // Lanes of vector g that lie in the window.
  auto lanes_of = [&](uint32_t g) {
    uint32_t l = 0xFu;
    if (g == 0) l &= (0xFu << lead) & 0xFu;
    if (g == ffull) l &= (1u << tailn) - 1u;
    return l;
  };

  // ---------------------------------------------------------------- guess: block64 samples
  // (from global memory, in flight together with the copies).  Start of run b =
  // floor(b (nv - 64) / (nblk - 1)), one run per lane (nblk <= 32), shuffled to the samples' lanes.
  const uint32_t nsamp = sample_count(uint32_t(k), nv, 8u);
  const uint32_t nblk = nsamp >> 6;
  const uint32_t sq = (nv - 64u) / (nblk - 1u), sr = (nv - 64u) % (nblk - 1u);
  const uint32_t run_start = uint32_t(lane) * sq + (uint32_t(lane) * sr) / (nblk - 1u);
  float sv[KPT];
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const uint32_t i = uint32_t(q * T + tid);
    const uint32_t s0 = __shfl_sync(FULL_MASK, run_start, (i >> 6) & 31u);
    sv[q] = i < nsamp ? __ldg(rowp + a + s0 + (i & 63u)) : qnan;
  }
  if (tid == 0) {
    mbar_init(&S.bar, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&S.bar, ffull * 16u);
    for (uint32_t c = 0; c < ffull; c += SHORT_COPY_VEC) {
      const uint32_t n = ffull - c < SHORT_COPY_VEC ? ffull - c : SHORT_COPY_VEC;
      bulk_copy_g2s(rv + c, base + 4 * size_t(c), n * 16u, &S.bar);
    }
  }
  for (int i = tid; i < (NB + 4) / 4; i += T) reinterpret_cast<uint4*>(S.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) S.ctr_win = S.ctr_cand = S.ctr_tie = S.list_n = S.tout = 0;
  if (tid == 32 && tailn) {
    const float* q = base + 4 * size_t(ffull);
    rv[ffull] = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
  }
  float lmin = INFINITY, lmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < KPT; ++q)
    if (isfinite(sv[q])) {
      lmin = fminf(lmin, sv[q]);
      lmax = fmaxf(lmax, sv[q]);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lmin = fminf(lmin, __shfl_xor_sync(FULL_MASK, lmin, o));
    lmax = fmaxf(lmax, __shfl_xor_sync(FULL_MASK, lmax, o));
  }
  if (lane == 0) {
    S.wmin[warp] = lmin;
    S.wmax[warp] = lmax;
  }
  __syncthreads();  // also publishes the mbarrier's initialisation to every thread
  static_assert(NW == 32, "each lane reads one warp's sample bounds");
  float gmin = S.wmin[lane], gmax = S.wmax[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gmin = fminf(gmin, __shfl_xor_sync(FULL_MASK, gmin, o));
    gmax = fmaxf(gmax, __shfl_xor_sync(FULL_MASK, gmax, o));
  }
  gmin = __fadd_rn(gmin, 0.0f);  // -0 -> +0
  const bool bracket_ok = isfinite(gmin) && isfinite(gmax) && gmin < gmax && !(p.flags & FLAG_FORCE_RESCUE);
  // The sampled floor, as in the cluster kernel: the lower edge of the bin where
  // mu + 3 sqrt(mu) + 6 samples are reached (mu = k nsamp / nv), bins ending lower when a few far
  // samples stretch them; -FLT_MAX in the lowest bin.
  float sc = 1.0f, thr = -FLT_MAX;
  if (bracket_ok) {
    sc = __fdiv_rn(float(NB), __fsub_rn(gmax, gmin));
    const float mu = float(k) * float(nsamp) / float(nv);
    const float want_f = mu + 3.0f * sqrtf(mu) + 6.0f;
    const uint32_t want = want_f < float(nsamp) ? uint32_t(want_f) : nsamp;
#pragma unroll
    for (int q = 0; q < KPT; ++q)
      if (!isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
    __syncthreads();
    static_assert(T == NB, "thread t holds bin NB - 1 - t in the scans");
    int fb = NB - 1 - short_cross(S, S.hist[NB - 1 - tid], want).t;
    if (fb == NB) fb = -1;
    const float rf = mu - 4.0f * sqrtf(mu);
    int hb = -1;
    if (rf >= 2.0f && fb < NB / 2) {
      hb = NB - 1 - short_cross(S, S.hist[NB - 1 - tid], uint32_t(rf)).t;
      if (hb == NB) hb = -1;
    }
    if (hb >= 0 && hb < NB / 2) {
      const float hi = __fadd_rn(gmin, __fdiv_rn(float(hb + 1), sc));
      sc = __fdiv_rn(float(NB), __fsub_rn(hi, gmin));
      for (int i = tid; i < NB; i += T) S.hist[i] = 0;
      __syncthreads();
#pragma unroll
      for (int q = 0; q < KPT; ++q)
        if (!isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
      __syncthreads();
      fb = NB - 1 - short_cross(S, S.hist[NB - 1 - tid], want).t;
      if (fb == NB) fb = -1;
    }
    thr = fb > 0 ? __fadd_rn(gmin, __fdiv_rn(float(fb), sc)) : -FLT_MAX;
    for (int i = tid; i < NB + 4; i += T) S.hist[i] = 0;
  }

  // ---------------------------------------------------------------- wait for the window
  // Warp 0 waits on the copies' mbarrier; the CTA barrier passes what it saw on to the others.
  if (warp == 0 && !mbar_wait_bounded(&S.bar, 0, WAIT_LIMIT_NS)) S.tout = 1;
  // diagnostics: row 0 reports a give-up once its window has landed (no copy in flight)
  if (tid == 0 && (p.flags & FLAG_DIAG_FAIL_ROW0) && row == 0) S.tout = 1;
  __syncthreads();
  if (S.tout) {  // gave up: wait (bounded) for the copies still in flight, then mark the row
    if (tid == 0) mbar_wait_bounded(&S.bar, 0, WAIT_LIMIT_NS);
    __syncthreads();
    for (int i = tid; i < k; i += T) out[i] = -2;
    if (stats) {
      stats[0] = PATH_DEVICE_ERROR;
      stats[1] = stats[2] = stats[3] = 0;
    }
    return;
  }

  // ---------------------------------------------------------------- verify: list and histogram >= t
  // Each thread marks the scores of its vectors that reach the floor (bit 4i + l: lane l of its
  // i-th vector), takes list slots for them with one atomic per warp, lists their positions in
  // the staged vectors and counts them in the histogram; the collect then walks the list with
  // every lane busy.
  constexpr int VPT_MAX = (SHORT_MAX / 4 + 1 + T - 1) / T;  // vectors per thread at most
  static_assert(4 * VPT_MAX <= 32 && 4 * (SHORT_MAX / 4 + 1) <= 65536, "bit masks and 16-bit positions");
  const float* const rf = reinterpret_cast<const float*>(rv);
  bool decided = false;
  int32_t bstar = 0;
  uint32_t m = 0, above = 0, listed = 0;
  if (bracket_ok) {
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < VPT_MAX; ++i) {
      const uint32_t g = uint32_t(i * T + tid);
      if (g < nvec) {
        const float4 x = short_masked(rv[g], g, lead);
        bits |= (uint32_t(x.x >= thr) | uint32_t(x.y >= thr) << 1 | uint32_t(x.z >= thr) << 2 |
                 uint32_t(x.w >= thr) << 3)
                << (4 * i);
      }
    }
    uint32_t slot = warp_slots(&S.list_n, __popc(bits));
    while (bits) {  // list and count each marked score
      const uint32_t bt = uint32_t(__ffs(bits) - 1);
      bits &= bits - 1u;
      const uint32_t pos = 4u * ((bt >> 2) * uint32_t(T) + uint32_t(tid)) + (bt & 3u);
      if (slot < uint32_t(SHORT_LIST)) S.list[slot] = uint16_t(pos);
      ++slot;
      atomicAdd(&S.hist[value_bin(rf[pos], gmin, sc)], 1u);
    }
    __syncthreads();
    listed = S.list_n;
    if (listed <= uint32_t(SHORT_LIST)) {  // else the rescue below
      // the bin that crosses the k-th score (none when fewer than k scores reach the floor)
      const ShortCross cr = short_cross(S, S.hist[NB - 1 - tid], uint32_t(k));
      if (cr.t >= 0) {
        bstar = NB - 1 - cr.t;
        above = cr.before;
        m = cr.at;
        decided = m <= uint32_t(SHORT_CAND);
      }
    }
  }
  if (decided) {
    // -------------------------------------------------------------- refine
    const uint32_t need = uint32_t(k) - above;
    // Winners (above the crossing bin) straight to the output, the crossing bin's members' positions
    // to the candidate buffer: one ballot and one atomic per warp and kind.
    for (uint32_t i0 = 0; i0 < listed; i0 += T) {
      const uint32_t i = i0 + tid;
      const bool in = i < listed;
      const uint32_t pos = in ? S.list[i] : 0u;
      const float e = rf[pos];
      const int b = in ? value_bin(e, gmin, sc) : -1;
      const bool win = b > bstar, cand = in && b == bstar;
      const uint32_t w = warp_alloc_local(&S.ctr_win, win);
      if (win && w < above) {
        out[w] = int32_t(pos) - int32_t(lead);
        if (outv) outv[w] = e;
      }
      const uint32_t c = warp_alloc_local(&S.ctr_cand, cand);
      if (cand && c < uint32_t(SHORT_CAND)) S.cand[c] = uint16_t(pos);
    }
    __syncthreads();
    if (m <= uint32_t(RANK_REFINE_MAX)) {
      // rank of candidate i = candidates ordered before it by (value desc, index asc); positions
      // are in index order
      for (uint32_t i = tid; i < m; i += T) {
        const uint32_t pi = S.cand[i];
        const float cv = rf[pi];
        uint32_t r = 0;
        for (uint32_t q = 0; q < m; ++q) {
          const uint32_t pq = S.cand[q];
          const float w = rf[pq];
          r += (w > cv) || (w == cv && pq < pi);
        }
        if (r < need) {
          out[above + r] = int32_t(pi) - int32_t(lead);
          if (outv) outv[above + r] = cv;
        }
      }
    } else {
      // radix select of the need largest order keys among the candidates, 8 bits a pass
      uint32_t prefix = 0, pmask = 0, rneed = need;
      bool ge = false;
      for (int shift = 24; shift >= 0; shift -= 8) {
        __syncthreads();
        for (int i = tid; i < 256; i += T) S.hist[i] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < m; i += T) {
          const uint32_t key = order_key(rf[S.cand[i]]);
          if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        const ShortCross dc = short_cross(S, tid < 256 ? S.hist[255 - tid] : 0u, rneed);
        prefix |= uint32_t(255 - dc.t) << shift;
        pmask |= 0xFFu << shift;
        rneed -= dc.before;
        if (dc.at == rneed) {
          ge = true;
          break;
        }
      }
      const uint32_t nties = ge ? 0u : rneed;
      const uint32_t tie_base = above + (need - nties);
      for (uint32_t b0 = 0; b0 < m; b0 += T) {
        const uint32_t i = b0 + tid;
        const bool in = i < m;
        const uint32_t pi = in ? S.cand[i] : 0u;
        const float cv = rf[pi];
        const uint32_t key = order_key(cv);
        const bool win = in && (ge ? (key & pmask) >= prefix : key > prefix);
        const bool tie = in && !ge && key == prefix;
        const uint32_t w = warp_alloc_local(&S.ctr_win, win);
        if (win && w < tie_base) {
          out[w] = int32_t(pi) - int32_t(lead);
          if (outv) outv[w] = cv;
        }
        const uint32_t t = warp_alloc_local(&S.ctr_tie, tie);
        if (tie && t < nties) {
          out[tie_base + t] = int32_t(pi) - int32_t(lead);
          if (outv) outv[tie_base + t] = cv;
        }
      }
    }
    if (stats) {
      stats[0] = PATH_SHORT_KERNEL;
      stats[1] = int32_t(m);
      stats[2] = 1;
      stats[3] = int32_t(above);
    }
    return;
  }

  // ---------------------------------------------------------------- rescue: radix over the row
  // Exact selection over the order keys of the resident window, one 8-bit digit a pass from the
  // top, stopping once the keys above the chosen digit are exactly the ones still needed or every
  // remaining key is equal; then one emission pass.
  uint32_t prefix = 0, pmask = 0, rneed = uint32_t(k);
  bool ge = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    __syncthreads();
    for (int i = tid; i < 256; i += T) S.hist[i] = 0;
    if (tid == 0) {
      S.kmin_loc = 0xffffffffu;
      S.kmax_loc = 0u;
    }
    __syncthreads();
    uint32_t tmin = 0xffffffffu, tmax = 0u;
    for (uint32_t g = tid; g < nvec; g += T) {
      const float4 x = rv[g];
      const uint32_t ln = lanes_of(g);
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const uint32_t key = order_key(f4_get(x, l));
        if (((ln >> l) & 1u) && (key & pmask) == prefix) {
          atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
          tmin = min(tmin, key);
          tmax = max(tmax, key);
        }
      }
    }
    tmin = __reduce_min_sync(FULL_MASK, tmin);
    tmax = __reduce_max_sync(FULL_MASK, tmax);
    if (lane == 0) {
      atomicMin(&S.kmin_loc, tmin);
      atomicMax(&S.kmax_loc, tmax);
    }
    __syncthreads();
    if (S.kmin_loc == S.kmax_loc) {  // every remaining key is the same: ties
      prefix = S.kmin_loc;
      pmask = 0xffffffffu;
      break;
    }
    const ShortCross dc = short_cross(S, tid < 256 ? S.hist[255 - tid] : 0u, rneed);
    prefix |= uint32_t(255 - dc.t) << shift;
    pmask |= 0xFFu << shift;
    rneed -= dc.before;
    if (dc.at == rneed) {
      ge = true;
      break;
    }
  }
  const uint32_t nties = ge ? 0u : rneed;
  const uint32_t tie_base = uint32_t(k) - nties;
  uint32_t nw = 0, nt = 0;
  for (uint32_t g = tid; g < nvec; g += T) {
    const float4 x = rv[g];
    const uint32_t ln = lanes_of(g);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const uint32_t key = order_key(f4_get(x, l));
      const bool valid = (ln >> l) & 1u;
      nw += valid && (ge ? (key & pmask) >= prefix : key > prefix);
      nt += valid && !ge && key == prefix;
    }
  }
  uint32_t ws, ts;
  warp_slots2(&S.ctr_win, &S.ctr_tie, nw, nt, ws, ts);
  if ((nw && ws < tie_base) || (nt && ts < nties)) {
    for (uint32_t g = tid; g < nvec; g += T) {
      const float4 x = rv[g];
      const uint32_t ln = lanes_of(g);
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const float e = f4_get(x, l);
        const uint32_t key = order_key(e);
        const bool valid = (ln >> l) & 1u;
        const int32_t jw = int32_t(4 * g + l) - int32_t(lead);
        if (valid && (ge ? (key & pmask) >= prefix : key > prefix)) {
          if (ws < tie_base) {
            out[ws] = jw;
            if (outv) outv[ws] = e;
          }
          ++ws;
        } else if (valid && !ge && key == prefix) {
          if (ts < nties) {
            out[tie_base + ts] = jw;
            if (outv) outv[tie_base + ts] = e;
          }
          ++ts;
        }
      }
    }
  }
  if (stats) {
    stats[0] = PATH_SHORT_KERNEL_RADIX;
    stats[1] = int32_t(m);
    stats[2] = 1;
    stats[3] = 0;
  }
}

}  // namespace gvr
