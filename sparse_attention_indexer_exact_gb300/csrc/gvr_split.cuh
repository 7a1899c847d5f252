// gvr_split.cuh -- the balanced GVR top-K kernel: rows of uneven length split into equal chunks.
//
// The cluster kernel (gvr_kernel.cuh) gives every row the same number of CTAs, chosen on the
// host from the row stride, because the real row lengths (from kv_lens or the window bounds)
// live on the device.  In a decode batch whose lengths spread from a few thousand to the full
// stride, the CTAs of the longest rows then set the launch time while the others idle.  This
// kernel decides the split on the device instead: every CTA reads all rows' lengths, cuts the
// batch's valid scores into chunks of one common size (rounded to whole 4 KB stages), and takes
// the chunk whose number is its block index.  Per chunk, the GVR steps of "GVR K=2048 reg_clus
// with block64 sampling and parallel rescue" (TensorRT-LLM PR #20998, "What changes") run as:
//
//   Guess   the row's uniform block64 samples (the same positions and count as the cluster
//           kernel) give GMIN / GMAX and the sampled floor t, identically in every chunk of the
//           row (same samples, same arithmetic);
//   Verify  the chunk streams through a shared-memory ring filled by bulk copies; every score
//           >= t (a few per cent of the row) is published to the chunk's slot of the workspace;
//   Refine  the last chunk of the row to finish (a per-row arrival counter) reads the row's
//           published scores from L2, histograms them over the value bins of [GMIN, GMAX],
//           finds the bin that crosses the K-th largest score ("Why the GLM row overflows"),
//           writes the winners above it and refines the crossing bin's members exactly.
//
// Exactness: every score of the row that is >= t was published, so when at least K were, the
// K largest of the row are the K largest of the published ones.  When fewer than K reached t, a
// chunk overflowed its slot, or the crossing bin holds more members than the idle ring can take,
// the last CTA selects the row alone by an exact radix select over the order keys of the whole
// window (4 digit passes at most, reading the row from global memory) -- correct in every case,
// slow for long rows, and rare: the floor's margin makes it a per-row event of about 1e-4 on the
// workloads' score distributions.
//
// The workspace (caller-owned, zero-filled before its first use) holds per chunk the published
// scores and window indices and their count, and per row the arrival counter; the last chunk of
// a row resets that counter, so every call leaves the workspace as it found it.
#pragma once

#include "gvr_kernel.cuh"

namespace gvr {

constexpr int SPLIT_NST = 6;                 // ring stages (4 KB each) per CTA
constexpr int SPLIT_CTAS_PER_SM = 6;         // occupancy the launch bound and shared memory allow
constexpr int SPLIT_UNIT_CAP = 4096;         // scores one chunk can publish
constexpr int32_t SPLIT_MIN_CHUNK_VEC = 1024;  // 4096 scores: the smallest chunk
constexpr int SPLIT_MAX_ROWS = 512;          // rows a split launch can schedule
constexpr int SPLIT_MAX_UNITS_ROW = 256;     // chunks of one row the last CTA gathers in shared memory
constexpr int SPLIT_STASH = 4096;            // published (score, index) pairs it gathers at most
constexpr int FB = 256;                      // bins of the last CTA's histogram of the gathered scores
constexpr int PATH_SPLIT = 7;                // row_stats: selected from the published scores
constexpr int PATH_SPLIT_ALONE = 8;          // row_stats: the last CTA selected the row alone

enum : int32_t { FLAG_SPLIT_ALONE = 512 };   // diagnostics: every long row takes the lone path

struct SplitParams {
  const float* logits;
  int64_t row_stride;
  const int32_t* kv_lens;     // decode
  const int32_t* row_starts;  // prefill
  const int32_t* row_ends;    // prefill
  int32_t* indices;
  float* values;              // nullable
  int32_t* row_stats;         // nullable, [rows][4]
  float* surv_v;              // workspace: [grid][SPLIT_UNIT_CAP] published scores
  int32_t* surv_j;            // workspace: [grid][SPLIT_UNIT_CAP] their window indices
  uint32_t* surv_n;           // workspace: [grid] scores each chunk found >= t (may exceed the cap)
  uint32_t* arrive;           // workspace: [rows] chunks of the row done (zero between calls)
  int32_t num_rows;
  int32_t next_n;
  int32_t compress_ratio;
  int32_t k;
  int32_t mode;
  int32_t flags;
};

struct alignas(16) SplitSmem {
  uint32_t fh[FB + 4];                    // the last CTA: histogram / digit counts of the gathered scores
  uint32_t cnt[SPLIT_MAX_UNITS_ROW];      // the last CTA: each chunk's published count
  uint32_t off[SPLIT_MAX_UNITS_ROW + 1];  // ... and its first slot in the gathered arrays
  uint32_t wsum[2][8];
  float wmin[8], wmax[8];
  Crossing cross;
  float vthr;
  int32_t fpart;
  uint32_t dsel, dabove, dcnt, dmy_above, dmy_at;
  uint32_t kmin_loc, kmax_loc;
  uint32_t nsurv;                    // scores of this chunk >= t (may exceed SPLIT_UNIT_CAP)
  uint32_t ctr_win, ctr_cand, ctr_rwin, ctr_rtie;
  uint32_t red_n, red_over;          // the last CTA: published scores of the row, overflow flag
  int32_t sched[7];                  // row, chunk, chunks of the row, first chunk, all chunks, a, nv
  uint32_t is_last;
  uint32_t tout;
  uint32_t gather_n;                 // the last CTA: gathered slots (chunks padded to 4 entries)
  float gvmin, gvmax;                // the last CTA: range of the gathered scores
  float4 tail;
  uint64_t bar[SPLIT_NST];
  uint64_t fbar;                     // the last CTA: the gathering copies have landed
  // Last members: hist, tot and the ring after them form one contiguous area, which the last
  // CTA reuses to gather the row's published pairs (values first, then indices).
  alignas(16) uint32_t hist[NB + 4];  // the samples' histogram (floor)
  union {
    uint32_t tot[NB + 4];  // (space: part of the last CTA's gathering area)
    struct {               // the schedule: every row's window
      uint32_t nv[SPLIT_MAX_ROWS];
      uint32_t a[SPLIT_MAX_ROWS];
    } rows;
  };
};
static_assert(offsetof(SplitSmem, hist) % 16 == 0 && offsetof(SplitSmem, tot) % 16 == 0,
              "histograms are read as 16-byte vectors");
static_assert(offsetof(SplitSmem, bar) % 8 == 0 && offsetof(SplitSmem, fbar) % 8 == 0,
              "mbarriers must be 8-byte aligned");
static_assert(2 * SPLIT_MAX_ROWS <= NB + 4, "the schedule fits the histogram it shares memory with");

constexpr int SPLIT_SMEM_FIXED = int((sizeof(SplitSmem) + 127) / 128 * 128);
__host__ __device__ constexpr int split_smem_bytes() { return SPLIT_SMEM_FIXED + SPLIT_NST * STAGE_VEC * 16; }
static_assert(split_smem_bytes() - int(offsetof(SplitSmem, hist)) >= 8 * SPLIT_STASH,
              "hist, tot and the ring hold the gathered pairs");

// Window [a, a + nv) of row r (the same geometry as the cluster kernel's head) from its inputs:
// decode x = kv_lens[r / next_n]; prefill x = row_starts[r], y = row_ends[r].
__device__ __forceinline__ void split_row_window(const SplitParams& p, uint32_t r, int32_t x, int32_t y, uint32_t& a,
                                                 uint32_t& nv) {
  const uint32_t stride = uint32_t(p.row_stride);
  a = 0;
  nv = 0;
  if (p.mode == MODE_DECODE) {
    const uint32_t nn = uint32_t(p.next_n);
    const uint32_t req = r / nn;
    const int32_t kv = x;
    if (kv >= p.next_n) nv = (uint32_t(kv) - nn + (r - req * nn) + 1u) / uint32_t(p.compress_ratio);
    nv = nv < stride ? nv : stride;
  } else {
    const int32_t ks = x;
    const int32_t ke = y;
    const uint32_t s = ks > 0 ? uint32_t(ks) : 0u;
    const uint32_t e = ke > 0 ? (uint32_t(ke) < stride ? uint32_t(ke) : stride) : 0u;
    a = s < stride ? s : stride;
    nv = e > a ? e - a : 0u;
  }
}

// Chunks of a row: one for a short row (it writes the identity), else its vectors over the
// chunk size.
__device__ __forceinline__ uint32_t split_units(uint32_t a, uint32_t nv, uint32_t k, uint32_t chv) {
  if (nv <= k) return 1u;
  const uint32_t nvec = ((a & 3u) + nv + 3u) >> 2;
  return (nvec + chv - 1u) / chv;
}

template <bool UNUSED>
__global__ void __launch_bounds__(THREADS, SPLIT_CTAS_PER_SM) gvr_split_kernel(const SplitParams p) {
  constexpr int T = THREADS;
  constexpr int NW = T / 32;
  constexpr int KPT = (MAX_K + T - 1) / T;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SplitSmem& S = *reinterpret_cast<SplitSmem*>(smem_raw);
  float4 (*ring)[STAGE_VEC] = reinterpret_cast<float4 (*)[STAGE_VEC]>(smem_raw + SPLIT_SMEM_FIXED);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t k = p.k;
  const int32_t R = p.num_rows;
  const uint32_t unit = blockIdx.x;
  const float qnan = __int_as_float(0x7fffffff);

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < SPLIT_NST; ++s) mbar_init(&S.bar[s], 1);
    mbar_init(&S.fbar, 1);
    mbar_init_fence();
  }

  // ---------------------------------------------------------------- schedule (warp 0)
  // Every CTA computes the same split: rows' windows, the chunk size (the long rows' vectors
  // over the grid minus one chunk per row for rounding, whole stages, at least
  // SPLIT_MIN_CHUNK_VEC), the chunks of each row in row order, and which chunk is this block's.
  if (warp == 0) {
    uint64_t fsum = 0;
    for (int32_t r0 = 0; r0 < R; r0 += 4 * 32) {  // four rows per lane in flight at once
      int32_t x[4], y[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int32_t r = r0 + 32 * q + lane;
        x[q] = y[q] = 0;
        if (r < R) {
          if (p.mode == MODE_DECODE) {
            x[q] = __ldg(p.kv_lens + uint32_t(r) / uint32_t(p.next_n));
          } else {
            x[q] = __ldg(p.row_starts + r);
            y[q] = __ldg(p.row_ends + r);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int32_t r = r0 + 32 * q + lane;
        if (r < R) {
          uint32_t a, nv;
          split_row_window(p, uint32_t(r), x[q], y[q], a, nv);
          S.rows.a[r] = a;
          S.rows.nv[r] = nv;
          if (nv > uint32_t(k)) fsum += ((a & 3u) + nv + 3u) >> 2;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fsum += __shfl_xor_sync(FULL_MASK, fsum, o);
    __syncwarp();
    const uint64_t denom = uint64_t(gridDim.x) - uint64_t(R);  // the host keeps the grid >= 2 rows
    uint64_t chv = (fsum + denom - 1u) / denom;
    chv = (chv + STAGE_VEC - 1) / STAGE_VEC * STAGE_VEC;
    if (chv < uint64_t(SPLIT_MIN_CHUNK_VEC)) chv = SPLIT_MIN_CHUNK_VEC;
    const uint32_t cv = uint32_t(chv);  // <= the longest row's vectors rounded up: < 2^30
    const int32_t per = (R + 31) / 32;  // rows [lane * per, lane * per + per) in row order
    const int32_t r0 = lane * per, r1 = min(R, r0 + per);
    uint32_t mine = 0;
    for (int32_t r = r0; r < r1; ++r) mine += split_units(S.rows.a[r], S.rows.nv[r], uint32_t(k), cv);
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t total = __shfl_sync(FULL_MASK, incl, 31);  // <= gridDim.x by the chunk size
    uint32_t base = incl - mine;
    if (unit >= base && unit < incl) {
      for (int32_t r = r0; r < r1; ++r) {
        const uint32_t nu = split_units(S.rows.a[r], S.rows.nv[r], uint32_t(k), cv);
        if (unit < base + nu) {
          S.sched[0] = r;
          S.sched[1] = int32_t(unit - base);
          S.sched[2] = int32_t(nu);
          S.sched[3] = int32_t(base);
          S.sched[5] = int32_t(S.rows.a[r]);
          S.sched[6] = int32_t(S.rows.nv[r]);
          break;
        }
        base += nu;
      }
    }
    if (lane == 0) {
      S.sched[4] = int32_t(total);
      S.vthr = __uint_as_float(cv);  // the chunk size, passed through shared memory
    }
  }
  __syncthreads();
  if (unit >= uint32_t(S.sched[4])) return;  // no chunk left for this block
  const uint32_t row = uint32_t(S.sched[0]);
  const int32_t chunk = S.sched[1];
  const int32_t nunits = S.sched[2];
  const uint32_t unit0 = uint32_t(S.sched[3]);
  const uint32_t a = uint32_t(S.sched[5]);
  const uint32_t nv = uint32_t(S.sched[6]);
  const int32_t chv = int32_t(__float_as_uint(S.vthr));
  const float* rowp = p.logits + int64_t(row) * p.row_stride;
  int32_t* out = p.indices + int64_t(row) * k;
  float* outv = p.values ? p.values + int64_t(row) * k : nullptr;

  // ---------------------------------------------------------------- short row: identity
  if (nv <= uint32_t(k)) {
    for (int i = tid; i < k; i += T) {
      out[i] = uint32_t(i) < nv ? i : -1;
      if (outv) outv[i] = uint32_t(i) < nv ? rowp[a + i] : -FLT_MAX;
    }
    if (p.row_stats && tid == 0) {
      int32_t* st = p.row_stats + 4 * int64_t(row);
      st[0] = PATH_SHORT;
      st[1] = st[2] = st[3] = 0;
    }
    return;
  }

  // ---------------------------------------------------------------- this chunk's vectors
  // Vectors are 16-byte aligned float4s from the aligned column at or below the window start
  // (vector g holds window positions 4g - lead .. 4g + 3 - lead); the chunk is vectors
  // [v0, v1) of the window, streamed in stages of STAGE_VEC vectors.
  const int32_t lead = int32_t(a & 3u);
  const float* base = rowp + (a - uint32_t(lead));
  const int32_t span = lead + int32_t(nv);
  const int32_t ffull = span >> 2;
  const int32_t tailn = span & 3;
  const int32_t nvec = ffull + (tailn ? 1 : 0);
  const int32_t v0 = chunk * chv;
  const int32_t v1 = min(nvec, v0 + chv);
  const int32_t nst = (v1 - v0 + STAGE_VEC - 1) / STAGE_VEC;
  auto issue_stage = [&](int32_t s, uint32_t slot) {  // one thread
    const int32_t c0 = v0 + s * STAGE_VEC;
    const int32_t c1 = min(min(c0 + STAGE_VEC, v1), ffull);
    if (c1 > c0) {
      mbar_arrive_expect_tx(&S.bar[slot], uint32_t(c1 - c0) * 16u);
      bulk_copy_g2s(&ring[slot][0], base + 4 * size_t(c0), uint32_t(c1 - c0) * 16u, &S.bar[slot]);
    } else {
      mbar_arrive(&S.bar[slot]);  // a stage holding only the partial last vector
    }
  };

  // ---------------------------------------------------------------- guess: block64 sample
  const uint32_t nsamp = sample_count(uint32_t(k), nv, 8u);
  const uint32_t nblk = nsamp >> 6;
  const uint32_t sq = (nv - 64u) / (nblk - 1u), sr = (nv - 64u) % (nblk - 1u);
  const uint32_t run_start = uint32_t(lane) * sq + (uint32_t(lane) * sr) / (nblk - 1u);
  float sv[KPT];
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const uint32_t i = uint32_t(q * T + tid);
    const uint32_t s = __shfl_sync(FULL_MASK, run_start, (i >> 6) & 31u);
    sv[q] = i < nsamp ? __ldg(rowp + a + s + (i & 63u)) : qnan;
  }
  // the chunk's first stages go in flight right behind the samples
  if (warp == 0 && lane < SPLIT_NST && lane < nst) issue_stage(lane, uint32_t(lane));
  for (int i = tid; i < NB + 4; i += T) S.hist[i] = 0;
  if (tid == 0) {
    S.nsurv = 0;
    S.tout = 0;
  }
  if (tid == 32) {  // the partial last vector, read with scalar loads, never past the window
    S.tail = make_float4(qnan, qnan, qnan, qnan);
    if (tailn && ffull >= v0 && ffull < v1) {
      const float* q = base + 4 * size_t(ffull);
      S.tail = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
    }
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
  __syncthreads();
  float gmin = INFINITY, gmax = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    gmin = fminf(gmin, S.wmin[w]);
    gmax = fmaxf(gmax, S.wmax[w]);
  }
  gmin = __fadd_rn(gmin, 0.0f);  // -0 -> +0
  const bool bracket_ok = isfinite(gmin) && isfinite(gmax) && gmin < gmax;
  // The samples have landed (every thread is past the barrier above): ask L2 for the rest of
  // the chunk beyond the ring's first stages, so the refills later find it there.
  if (tid == 0 && nst > SPLIT_NST) {
    const int32_t c0 = v0 + SPLIT_NST * STAGE_VEC, c1 = min(v1, ffull);
    if (c1 > c0) bulk_prefetch_l2(base + 4 * size_t(c0), uint32_t(c1 - c0) * 16u);
  }
  // The sampled floor, as in the cluster kernel: the lower edge of the bin where
  // mu + 3 sqrt(mu) + 6 samples are reached (mu = k nsamp / nv, the samples expected above
  // tau), with the bins ending lower when a few far samples stretch them.
  float sc = 1.0f;
  float thr = -INFINITY;
  if (bracket_ok) {
    sc = __fdiv_rn(float(NB), __fsub_rn(gmax, gmin));
    const float mu = float(k) * float(nsamp) / float(nv);
    const float want_f = mu + 3.0f * sqrtf(mu) + 6.0f;
    const uint32_t want = want_f < float(nsamp) ? uint32_t(want_f) : nsamp;
#pragma unroll
    for (int q = 0; q < KPT; ++q)
      if (!isnan(sv[q])) atomicAdd(&S.hist[value_bin(sv[q], gmin, sc)], 1u);
    __syncthreads();
    int fb = suffix_cross<T>(S, S.hist, want);
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
    thr = fb > 0 ? __fadd_rn(gmin, __fdiv_rn(float(fb), sc)) : -INFINITY;
  }
  const bool alone = (p.flags & FLAG_SPLIT_ALONE) != 0;

  // ---------------------------------------------------------------- verify: publish >= t
  // One compare against the floor per score (a thread first takes the max of its 8 scores of
  // the stage); a thread with scores at or above it takes their slots with one shared atomic;
  // the published (score, window index) pairs go straight to the chunk's slot of the workspace.
  float* const my_v = p.surv_v + size_t(unit) * SPLIT_UNIT_CAP;
  int32_t* const my_j = p.surv_j + size_t(unit) * SPLIT_UNIT_CAP;
  bool late = false;
  for (int32_t s = 0; s < nst; ++s) {
    const uint32_t slot = uint32_t(s) % SPLIT_NST;
    const uint32_t ph = (uint32_t(s) / SPLIT_NST) & 1u;
    if (!mbar_wait_bounded(&S.bar[slot], ph, WAIT_LIMIT_NS)) {
      mbar_wait_bounded(&S.bar[slot], ph, WAIT_LIMIT_NS);  // let copies land
      late = true;
    }
    const int32_t c0 = v0 + s * STAGE_VEC;
    float4 vv[VPS];
    uint32_t lanes = 0xFFFFFFFFu;  // bit 4i+l: lane l of the i-th vector is in the window
    if (c0 > 0 && c0 + STAGE_VEC <= min(v1, ffull)) {  // an interior stage
#pragma unroll
      for (int i = 0; i < VPS; ++i) vv[i] = ring[slot][i * T + tid];
    } else {
      lanes = 0;
#pragma unroll
      for (int i = 0; i < VPS; ++i) {
        const int32_t g = c0 + i * T + tid;
        uint32_t ln = 0;
        vv[i] = f4_zero();
        if (g < v1) {
          if (g < ffull) {
            vv[i] = ring[slot][i * T + tid];
            ln = 0xFu;
          } else {
            vv[i] = S.tail;
            ln = (1u << tailn) - 1u;
          }
          if (g == 0) ln &= (0xFu << lead) & 0xFu;
        }
        lanes |= ln << (4 * i);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPS; ++i) mx = fmaxf(mx, fmaxf(fmaxf(vv[i].x, vv[i].y), fmaxf(vv[i].z, vv[i].w)));
    uint32_t bits = 0;
    if (mx >= thr) {
#pragma unroll
      for (int i = 0; i < VPS; ++i)
        bits |= (uint32_t(vv[i].x >= thr) | (uint32_t(vv[i].y >= thr) << 1) | (uint32_t(vv[i].z >= thr) << 2) |
                 (uint32_t(vv[i].w >= thr) << 3))
                << (4 * i);
      bits &= lanes;
    }
    static_assert(VPS == 2, "a stage's hit j lies in the thread's first or last vector");
    if (bits) {  // no warp collective: the thread's slots with one shared atomic
      uint32_t at = atomicAdd(&S.nsurv, uint32_t(__popc(bits)));
      if (!alone)
        for (; bits; bits &= bits - 1u, ++at) {
          const int j = __ffs(bits) - 1;
          if (at < uint32_t(SPLIT_UNIT_CAP)) {
            const float4 v = (j >> 2) == 0 ? vv[0] : vv[VPS - 1];
            my_v[at] = f4_get(v, j & 3);
            my_j[at] = 4 * (c0 + (j >> 2) * T + tid) - lead + (j & 3);
          }
        }
    }
    if (s + SPLIT_NST < nst) {  // refill this slot once every thread is done with it
      if (__syncthreads_or(late)) {
        // drain the stages already in flight, then stop: the row is marked failed
        for (int32_t d = s + 1; d < nst && d < s + SPLIT_NST; ++d)
          mbar_wait_bounded(&S.bar[uint32_t(d) % SPLIT_NST], (uint32_t(d) / SPLIT_NST) & 1u, WAIT_LIMIT_NS);
        late = true;
        break;
      }
      if (tid == 0) issue_stage(s + SPLIT_NST, slot);
    }
  }
  if (__syncthreads_or(late) && tid == 0) S.tout = 1;

  // ---------------------------------------------------------------- publish, last chunk refines
  // The CTA barrier orders every thread's published pairs before thread 0's fence, and the fence
  // (cumulative) orders them before the count and the arrival: one device-scope fence per CTA.
  __syncthreads();
  if (tid == 0) {
    p.surv_n[unit] = S.tout ? 0xffffffffu : S.nsurv;  // a failed chunk marks the row
    __threadfence();
    const uint32_t old = atomicAdd(p.arrive + row, 1u);
    const bool last = old + 1u == uint32_t(nunits);
    if (last) {
      __threadfence();    // the other chunks' pairs and counts, published before their arrivals
      p.arrive[row] = 0;  // every chunk of the row has arrived: reset for the next call
    }
    S.is_last = last;
  }
  __syncthreads();
  if (!S.is_last) return;

  // ------------------------------------------------------------ gather the row's published pairs
  // Chunk q of the row published min(n_q, cap) pairs.  The last CTA copies them into its shared
  // memory (hist, tot and the idle ring: values first, then indices) with bulk copies, each
  // chunk at a 4-entry boundary (its last slots padded and marked with index -1).
  float* const gv = reinterpret_cast<float*>(&S.hist[0]);
  int32_t* const gj = reinterpret_cast<int32_t*>(&S.hist[0]) + SPLIT_STASH;
  if (tid == 0) {
    S.red_n = 0;
    S.red_over = 0;
    S.ctr_win = S.ctr_cand = 0;  // slot counters of the lone path
  }
  __syncthreads();
  const bool gatherable = nunits <= SPLIT_MAX_UNITS_ROW;
  if (gatherable) {
    for (int32_t q = tid; q < nunits; q += T) {
      const uint32_t n = __ldcg(p.surv_n + unit0 + q);
      S.cnt[q] = n;
      atomicAdd(&S.red_n, n < uint32_t(SPLIT_UNIT_CAP) ? n : uint32_t(SPLIT_UNIT_CAP));
      if (n > uint32_t(SPLIT_UNIT_CAP)) atomicOr(&S.red_over, n == 0xffffffffu ? 2u : 1u);
    }
    __syncthreads();
    if (warp == 0) {  // slots: each chunk's count rounded up to 4, in chunk order
      uint32_t run = 0;
      for (int32_t q0 = 0; q0 < nunits; q0 += 32) {
        const int32_t q = q0 + lane;
        const uint32_t n = q < nunits ? min(S.cnt[q], uint32_t(SPLIT_UNIT_CAP)) : 0u;
        const uint32_t r4 = (n + 3u) & ~3u;
        uint32_t incl = r4;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t x = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += x;
        }
        if (q < nunits) S.off[q] = run + incl - r4;
        run += __shfl_sync(FULL_MASK, incl, 31);
      }
      if (lane == 0) {
        S.off[nunits] = run;
        S.gather_n = run;
      }
    }
  } else if (tid == 0) {
    S.red_over = 1;  // more chunks than the last CTA gathers: the row is selected alone
  }
  __syncthreads();
  const uint32_t total = S.red_n;
  const bool failed = (S.red_over & 2u) != 0;
  const uint32_t gn = gatherable ? S.gather_n : 0u;
  bool ok = !failed && !alone && S.red_over == 0 && total >= uint32_t(k) && gn <= uint32_t(SPLIT_STASH);
  if (ok) {
    if (warp == 0) {
      if (lane == 0) {
        fence_proxy_async_global();  // the pairs were published by other CTAs' plain stores
        mbar_arrive_expect_tx(&S.fbar, gn * 8u);
      }
      __syncwarp();
      for (int32_t q = lane; q < nunits; q += 32) {
        const uint32_t o = S.off[q], b = (S.off[q + 1] - o) * 4u;
        if (b) {
          const size_t src = size_t(unit0 + uint32_t(q)) * SPLIT_UNIT_CAP;
          fence_proxy_async_global();
          bulk_copy_g2s(gv + o, p.surv_v + src, b, &S.fbar);
          bulk_copy_g2s(gj + o, p.surv_j + src, b, &S.fbar);
        }
      }
    }
    if (!mbar_wait_bounded(&S.fbar, 0u, WAIT_LIMIT_NS)) {
      mbar_wait_bounded(&S.fbar, 0u, WAIT_LIMIT_NS);  // let copies land
      late = true;
    }
    if (__syncthreads_or(late)) ok = false;
  }
  const bool gave_up = late;
  Crossing cr{};
  if (ok) {
    for (int32_t q = tid; q < nunits; q += T)  // mark the padding slots
      for (uint32_t e = S.off[q] + min(S.cnt[q], uint32_t(SPLIT_UNIT_CAP)); e < S.off[q + 1]; ++e) gj[e] = -1;
    __syncthreads();
    // ---------------------------------------------------------- verify: histogram, crossing bin
    // FB bins over the gathered scores' own range [vmin, vmax] (monotone bin function).
    float lo = INFINITY, hi = -INFINITY;
    for (uint32_t e = tid; e < gn; e += T)
      if (gj[e] >= 0) {
        lo = fminf(lo, gv[e]);
        hi = fmaxf(hi, gv[e]);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(FULL_MASK, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(FULL_MASK, hi, o));
    }
    if (lane == 0) {
      S.wmin[warp] = lo;
      S.wmax[warp] = hi;
    }
    for (int i = tid; i < FB; i += T) S.fh[i] = 0;
    __syncthreads();
    lo = INFINITY;
    hi = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      lo = fminf(lo, S.wmin[w]);
      hi = fmaxf(hi, S.wmax[w]);
    }
    // NaN never reaches the floor; a range that is not finite (+inf / -inf scores) or empty puts
    // every score in bin 0, where the radix selection below decides them exactly
    const float fsc = (isfinite(lo) && isfinite(hi) && hi > lo) ? __fdiv_rn(float(FB), __fsub_rn(hi, lo)) : 0.f;
    auto fbin = [&](float v) -> uint32_t {
      float x = __fmul_rn(__fsub_rn(v, lo), fsc);
      x = fminf(fmaxf(x, 0.0f), float(FB - 1));
      return uint32_t(__float2int_rz(x));
    };
    for (uint32_t e = tid; e < gn; e += T)
      if (gj[e] >= 0) atomicAdd(&S.fh[fbin(gv[e])], 1u);
    __syncthreads();
    const DigitCross fc = digit_scan<T>(S, S.fh, S.fh, uint32_t(k));
    cr.bin = int32_t(fc.digit);
    cr.above = fc.above;
    cr.m = fc.cnt;
    __syncthreads();
    // ---------------------------------------------------------- refine: radix select in the bin
    // The need = k - above largest order keys among the crossing bin's members, 8 bits a pass,
    // stopping once the keys above the chosen digit are exactly the ones needed or every
    // remaining key is equal.
    const uint32_t bstar = fc.digit;
    // A crossing bin of at most SPLIT_MAX_UNITS_ROW members is listed once (their stash slots, in
    // the per-chunk counts, idle by now) with its smallest and largest key: the digit passes then
    // read only the members, below the key bytes they all share.
    const bool compact = cr.m <= uint32_t(SPLIT_MAX_UNITS_ROW);
    if (tid == 0) {
      S.kmin_loc = 0xffffffffu;
      S.kmax_loc = 0u;
    }
    __syncthreads();
    if (compact) {
      uint32_t tmin = 0xffffffffu, tmax = 0u;
      for (uint32_t e = tid; e < gn; e += T)
        if (gj[e] >= 0 && fbin(gv[e]) == bstar) {
          const uint32_t key = order_key(gv[e]);
          S.cnt[atomicAdd(&S.ctr_cand, 1u)] = e;  // at most cr.m of them
          tmin = min(tmin, key);
          tmax = max(tmax, key);
        }
      tmin = __reduce_min_sync(FULL_MASK, tmin);
      tmax = __reduce_max_sync(FULL_MASK, tmax);
      if (lane == 0) {
        atomicMin(&S.kmin_loc, tmin);
        atomicMax(&S.kmax_loc, tmax);
      }
      __syncthreads();
    }
    const uint32_t kmin0 = S.kmin_loc, kmax0 = S.kmax_loc;
    const int dfix = !compact ? 0 : (kmin0 == kmax0 ? 4 : __clz(kmin0 ^ kmax0) / 8);
    uint32_t prefix = dfix >= 4 ? kmin0 : (dfix > 0 ? kmin0 & (0xffffffffu << (32 - 8 * dfix)) : 0u);
    uint32_t pmask = dfix >= 4 ? 0xffffffffu : (dfix > 0 ? 0xffffffffu << (32 - 8 * dfix) : 0u);
    uint32_t rneed = uint32_t(k) - cr.above;
    bool ge = false;
    __syncthreads();  // every thread has read the bounds before they are reset below
    for (int shift = 24 - 8 * dfix; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += T) S.fh[i] = 0;
      if (tid == 0) {
        S.kmin_loc = 0xffffffffu;
        S.kmax_loc = 0u;
      }
      __syncthreads();
      uint32_t tmin = 0xffffffffu, tmax = 0u;
      auto count = [&](float v) {
        const uint32_t key = order_key(v);
        if ((key & pmask) == prefix) {
          atomicAdd(&S.fh[(key >> shift) & 255u], 1u);
          tmin = min(tmin, key);
          tmax = max(tmax, key);
        }
      };
      if (compact) {
        for (uint32_t i = tid; i < cr.m; i += T) count(gv[S.cnt[i]]);
      } else {
        for (uint32_t e = tid; e < gn; e += T)
          if (gj[e] >= 0 && fbin(gv[e]) == bstar) count(gv[e]);
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
        __syncthreads();
        break;
      }
      const DigitCross dc = digit_scan<T>(S, S.fh, S.fh, rneed);
      __syncthreads();
      prefix |= dc.digit << shift;
      pmask |= 0xFFu << shift;
      rneed -= dc.above;
      if (dc.cnt == rneed) {
        ge = true;
        break;
      }
    }
    // ---------------------------------------------------------- emit
    // Winners (bins above the crossing bin, or its keys above tau) and the first nties ties, each
    // thread's own in turn, at offsets from block-wide prefix sums (no per-score atomics).
    const uint32_t nties = ge ? 0u : rneed;
    const uint32_t tie_base = uint32_t(k) - nties;
    auto classify = [&](uint32_t e, bool& win, bool& tie) {
      win = tie = false;
      if (gj[e] < 0) return;
      const float v = gv[e];
      const uint32_t b = fbin(v);
      if (b > bstar) {
        win = true;
      } else if (b == bstar) {
        const uint32_t key = order_key(v);
        win = ge ? (key & pmask) >= prefix : key > prefix;
        tie = !ge && key == prefix;
      }
    };
    uint32_t nw = 0, nt = 0;
    for (uint32_t e = tid; e < gn; e += T) {
      bool win, tie;
      classify(e, win, tie);
      nw += win;
      nt += tie;
    }
    uint32_t iw = nw, it = nt;  // inclusive warp scans, then warp offsets
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t a = __shfl_up_sync(FULL_MASK, iw, o), b = __shfl_up_sync(FULL_MASK, it, o);
      if (lane >= o) {
        iw += a;
        it += b;
      }
    }
    if (lane == 31) {
      S.wsum[0][warp] = iw;
      S.wsum[1][warp] = it;
    }
    __syncthreads();
    uint32_t ws = iw - nw, ts = it - nt;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if (w < warp) {
        ws += S.wsum[0][w];
        ts += S.wsum[1][w];
      }
    for (uint32_t e = tid; e < gn; e += T) {
      bool win, tie;
      classify(e, win, tie);
      if (win) {
        if (ws < tie_base) {  // always: the winners are exactly k - nties
          out[ws] = gj[e];
          if (outv) outv[ws] = gv[e];
        }
        ++ws;
      } else if (tie) {
        if (ts < nties) {
          out[tie_base + ts] = gj[e];
          if (outv) outv[tie_base + ts] = gv[e];
        }
        ++ts;
      }
    }
    if (p.row_stats && tid == 0) {
      int32_t* st = p.row_stats + 4 * int64_t(row);
      st[0] = PATH_SPLIT;
      st[1] = int32_t(cr.m);
      st[2] = nunits;
      st[3] = int32_t(cr.above);
    }
    return;
  }
  if (failed || gave_up) {
    for (int i = tid; i < k; i += T) out[i] = -2;
    if (p.row_stats && tid == 0) {
      int32_t* st = p.row_stats + 4 * int64_t(row);
      st[0] = PATH_DEVICE_ERROR;
      st[1] = st[2] = st[3] = 0;
    }
    return;
  }

  // ---------------------------------------------------------------- the row alone
  // Exact radix select over the order keys of the whole window, one 8-bit digit per pass from
  // the top, stopping early when the keys above the chosen digit are exactly the ones still
  // needed or every matching key is equal; then one emission pass.  The window is read with
  // coalesced 16-byte loads (the lead lanes and the partial last vector masked by position).
  uint32_t* const dh = S.hist;
  auto each_window = [&](auto&& f) {  // f(value, window index, valid), warp-collective
    for (int32_t g0 = 0; g0 < nvec; g0 += 4 * T) {
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t g = g0 + i * T + tid;
        v[i] = g < ffull ? __ldg(reinterpret_cast<const float4*>(base) + g) : f4_zero();
        if (g == ffull && tailn) {
          const float* q = base + 4 * size_t(ffull);
          v[i] = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int32_t g = g0 + i * T + tid;
        uint32_t ln = g < ffull ? 0xFu : (g == ffull ? (1u << tailn) - 1u : 0u);
        if (g == 0) ln &= (0xFu << lead) & 0xFu;
#pragma unroll
        for (int l = 0; l < 4; ++l) f(f4_get(v[i], l), 4 * g + l - lead, ((ln >> l) & 1u) != 0);
      }
    }
  };
  uint32_t prefix = 0, pmask = 0, rneed = uint32_t(k);
  bool ge = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += T) dh[i] = 0;
    if (tid == 0) {
      S.kmin_loc = 0xffffffffu;
      S.kmax_loc = 0u;
    }
    __syncthreads();
    uint32_t tmin = 0xffffffffu, tmax = 0u;
    each_window([&](float e, int32_t, bool valid) {
      const uint32_t key = order_key(e);
      if (valid && (key & pmask) == prefix) {
        atomicAdd(&dh[(key >> shift) & 255u], 1u);
        tmin = min(tmin, key);
        tmax = max(tmax, key);
      }
    });
    tmin = __reduce_min_sync(FULL_MASK, tmin);
    tmax = __reduce_max_sync(FULL_MASK, tmax);
    if (lane == 0) {
      atomicMin(&S.kmin_loc, tmin);
      atomicMax(&S.kmax_loc, tmax);
    }
    __syncthreads();
    if (S.kmin_loc == S.kmax_loc) {  // every key with this prefix is the same: ties
      prefix = S.kmin_loc;
      pmask = 0xffffffffu;
      __syncthreads();
      break;
    }
    const DigitCross dc = digit_scan<T>(S, dh, dh, rneed);
    __syncthreads();
    prefix |= dc.digit << shift;
    pmask |= 0xFFu << shift;
    rneed -= dc.above;
    if (dc.cnt == rneed) {
      ge = true;
      break;
    }
  }
  const uint32_t nties = ge ? 0u : rneed;
  const uint32_t tie_base = uint32_t(k) - nties;
  each_window([&](float e, int32_t jw, bool valid) {
    const uint32_t key = order_key(e);
    const bool win = valid && (ge ? (key & pmask) >= prefix : key > prefix);
    const bool tie = valid && !ge && key == prefix;
    const uint32_t ws = warp_alloc_local(&S.ctr_win, win);
    if (win && ws < tie_base) {
      out[ws] = jw;
      if (outv) outv[ws] = e;
    }
    const uint32_t ts = warp_alloc_local(&S.ctr_cand, tie);
    if (tie && ts < nties) {
      out[tie_base + ts] = jw;
      if (outv) outv[tie_base + ts] = e;
    }
  });
  if (p.row_stats && tid == 0) {
    int32_t* st = p.row_stats + 4 * int64_t(row);
    st[0] = PATH_SPLIT_ALONE;
    st[1] = int32_t(total);
    st[2] = nunits;
    st[3] = 0;
  }
}

}  // namespace gvr
