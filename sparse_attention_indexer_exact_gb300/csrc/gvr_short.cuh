// gvr_short.cuh -- register-resident GVR top-K for short rows (row stride <= 16384 scores).
//
// The cluster kernel (gvr_kernel.cuh) streams a row through a small shared-memory ring so that
// rows of any length work; for a short row that costs a latency chain per ring stage and a
// cluster exchange.  Here one CTA of 256 threads takes a whole row and holds it in registers:
// every thread issues all of its 16-byte loads of the window at once (VPT vectors, so the row
// arrives in one round trip) while the block64 samples ("GVR K=2048 reg_clus with block64
// sampling and parallel rescue", TensorRT-LLM PR #20998, "What changes") are loaded and reduced to
// the bracket [GMIN, GMAX] and the sampled floor t.  Then every step works on the registers:
//
//   Verify  the scores >= t are counted in NB value bins of the bracket (shared memory) and a
//           suffix scan finds the bin that crosses the K-th largest score ("Why the GLM row
//           overflows");
//   Refine  the winners of the bins above it are written, the crossing bin's members gathered
//           and the k - above largest of them picked exactly (rank counting, or a radix select
//           on their order keys);
//   Rescue  an invalid bracket, fewer than k scores at or above t, or a crossing bin larger than
//           the gather buffer take an exact radix select over the order keys of the whole row,
//           still in registers (4 digit passes at most, early exits).
//
// No cluster, no ring, no distributed shared memory, a small code body: a short row costs its
// load, a few passes over registers and the writes.
#pragma once

#include "gvr_kernel.cuh"

namespace gvr {

constexpr int SHORT_THREADS = 256;
constexpr int SHORT_MAX = 16384;   // row stride (scores) the kernel holds: 16 float4 per thread
constexpr int SHORT_CAND = 2048;   // crossing-bin members it gathers at most
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
};

struct alignas(16) ShortSmem {
  uint32_t hist[NB + 4];   // samples' histogram, then the scores' histogram, then digit counts
  float cand_v[SHORT_CAND];
  int32_t cand_j[SHORT_CAND];
  uint32_t wsum[2][8];
  float wmin[8], wmax[8];
  uint32_t dsel, dabove, dcnt, dmy_above, dmy_at;
  uint32_t kmin_loc, kmax_loc;
  uint32_t total, above, ctr_win, ctr_cand, ctr_tie;
};
static_assert(offsetof(ShortSmem, hist) % 16 == 0, "histograms are read as 16-byte vectors");

constexpr int SHORT_SMEM = int((sizeof(ShortSmem) + 127) / 128 * 128);

// Vectors per thread for a row stride: the smallest of 4, 8, 16 that holds any window (a window
// inside a row of row_stride scores spans at most row_stride / 4 vectors from its aligned start).
__host__ __device__ constexpr int short_vpt(int64_t row_stride) {
  return row_stride <= 4 * 4 * SHORT_THREADS ? 4 : (row_stride <= 8 * 4 * SHORT_THREADS ? 8 : 16);
}

template <int VPT>
__global__ void __launch_bounds__(SHORT_THREADS) gvr_short_kernel(const ShortParams p) {
  constexpr int T = SHORT_THREADS;
  constexpr int NW = T / 32;
  constexpr int KPT = (MAX_K + T - 1) / T;  // samples per thread at most
  __shared__ ShortSmem S;
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

  // Block-wide exclusive prefix of two per-thread counts (winners, ties): each thread's first
  // slot of each kind.  Block-collective.
  auto block_prefix2 = [&](uint32_t nw, uint32_t nt, uint32_t& ws, uint32_t& ts) {
    uint32_t iw = nw, it = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(FULL_MASK, iw, o), y = __shfl_up_sync(FULL_MASK, it, o);
      if (lane >= o) {
        iw += x;
        it += y;
      }
    }
    __syncthreads();  // wsum is free
    if (lane == 31) {
      S.wsum[0][warp] = iw;
      S.wsum[1][warp] = it;
    }
    __syncthreads();
    ws = iw - nw;
    ts = it - nt;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if (w < warp) {
        ws += S.wsum[0][w];
        ts += S.wsum[1][w];
      }
  };

  // ---------------------------------------------------------------- guess: block64 samples
  // (issued first: the floor needs them before the row is needed)
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
  // ---------------------------------------------------------------- the row into registers
  // Vector g = i T + tid of the window holds positions 4g - lead .. 4g + 3 - lead; each thread
  // loads its VPT vectors at once (the partial last vector as scalars, never past the window).
  const int32_t lead = int32_t(a & 3u);
  const float* base = rowp + (a - uint32_t(lead));
  const int32_t span = lead + int32_t(nv);
  const int32_t ffull = span >> 2;
  const int32_t tailn = span & 3;
  float4 v[VPT];
  uint32_t ln[VPT];  // lanes of each vector that lie in the window
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int32_t g = i * T + tid;
    v[i] = g < ffull ? __ldg(reinterpret_cast<const float4*>(base) + g) : make_float4(qnan, qnan, qnan, qnan);
    uint32_t l = g < ffull ? 0xFu : 0u;
    if (g == ffull && tailn) {
      const float* q = base + 4 * size_t(ffull);
      v[i] = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
      l = (1u << tailn) - 1u;
    }
    if (g == 0) l &= (0xFu << lead) & 0xFu;
    ln[i] = l;
  }

  for (int i = tid; i < NB + 4; i += T) S.hist[i] = 0;
  if (tid == 0) S.total = S.above = S.ctr_win = S.ctr_cand = S.ctr_tie = 0;
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
    thr = fb > 0 ? __fadd_rn(gmin, __fdiv_rn(float(fb), sc)) : -FLT_MAX;
    for (int i = tid; i < NB + 4; i += T) S.hist[i] = 0;
    __syncthreads();
  }

  // ---------------------------------------------------------------- verify: histogram >= t
  bool decided = false;
  int32_t bstar = 0;
  uint32_t m = 0;
  if (bracket_ok) {
    uint32_t cnt = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const float e = f4_get(v[i], l);
        if (((ln[i] >> l) & 1u) && e >= thr) {
          atomicAdd(&S.hist[value_bin(e, gmin, sc)], 1u);
          ++cnt;
        }
      }
    cnt = __reduce_add_sync(FULL_MASK, cnt);
    if (lane == 0) atomicAdd(&S.total, cnt);
    __syncthreads();
    if (S.total >= uint32_t(k)) {
      bstar = suffix_cross<T>(S, S.hist, uint32_t(k));  // the bin that crosses the k-th score
      uint32_t ab = 0;
      for (int b = bstar + 1 + tid; b < NB; b += T) ab += S.hist[b];
      ab = __reduce_add_sync(FULL_MASK, ab);
      if (lane == 0) atomicAdd(&S.above, ab);
      __syncthreads();
      m = S.hist[bstar];
      decided = m <= uint32_t(SHORT_CAND);
    }
  }
  if (decided) {
    // -------------------------------------------------------------- refine
    const uint32_t above = S.above, need = uint32_t(k) - above;
    // class of each score: 2 above the crossing bin (a winner), 1 in it (a candidate), 0 neither
    uint32_t nw = 0, nc = 0;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const float e = f4_get(v[i], l);
        if (((ln[i] >> l) & 1u) && e >= thr) {
          const int b = value_bin(e, gmin, sc);
          nw += b > bstar;
          nc += b == bstar;
        }
      }
    uint32_t ws, cs;
    block_prefix2(nw, nc, ws, cs);
    if (nw + nc) {
#pragma unroll
      for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          const float e = f4_get(v[i], l);
          if (((ln[i] >> l) & 1u) && e >= thr) {
            const int b = value_bin(e, gmin, sc);
            const int32_t jw = 4 * (i * T + tid) + l - lead;
            if (b > bstar) {
              if (ws < above) {
                out[ws] = jw;
                if (outv) outv[ws] = e;
              }
              ++ws;
            } else if (b == bstar) {
              if (cs < uint32_t(SHORT_CAND)) {
                S.cand_v[cs] = e;
                S.cand_j[cs] = jw;
              }
              ++cs;
            }
          }
        }
    }
    __syncthreads();
    if (m <= uint32_t(RANK_REFINE_MAX)) {
      // rank of candidate i = candidates ordered before it by (value desc, index asc)
      for (uint32_t i = tid; i < m; i += T) {
        const float cv = S.cand_v[i];
        const int32_t j = S.cand_j[i];
        uint32_t r = 0;
        for (uint32_t q = 0; q < m; ++q) {
          const float w = S.cand_v[q];
          r += (w > cv) || (w == cv && S.cand_j[q] < j);
        }
        if (r < need) {
          out[above + r] = j;
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
          const uint32_t key = order_key(S.cand_v[i]);
          if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        const DigitCross dc = digit_scan<T>(S, S.hist, S.hist, rneed);
        prefix |= dc.digit << shift;
        pmask |= 0xFFu << shift;
        rneed -= dc.above;
        if (dc.cnt == rneed) {
          ge = true;
          break;
        }
      }
      const uint32_t nties = ge ? 0u : rneed;
      const uint32_t tie_base = above + (need - nties);
      for (uint32_t b0 = 0; b0 < m; b0 += T) {
        const uint32_t i = b0 + tid;
        const bool in = i < m;
        const uint32_t key = in ? order_key(S.cand_v[i]) : 0u;
        const bool win = in && (ge ? (key & pmask) >= prefix : key > prefix);
        const bool tie = in && !ge && key == prefix;
        const uint32_t ws = warp_alloc_local(&S.ctr_win, win);
        if (win && ws < tie_base) {
          out[ws] = S.cand_j[i];
          if (outv) outv[ws] = S.cand_v[i];
        }
        const uint32_t ts = warp_alloc_local(&S.ctr_tie, tie);
        if (tie && ts < nties) {
          out[tie_base + ts] = S.cand_j[i];
          if (outv) outv[tie_base + ts] = S.cand_v[i];
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
  // Exact selection over the order keys of the whole row in registers, one 8-bit digit a pass
  // from the top, stopping once the keys above the chosen digit are exactly the ones still
  // needed or every remaining key is equal; then one emission pass.
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
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const uint32_t key = order_key(f4_get(v[i], l));
        if (((ln[i] >> l) & 1u) && (key & pmask) == prefix) {
          atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
          tmin = min(tmin, key);
          tmax = max(tmax, key);
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
    const DigitCross dc = digit_scan<T>(S, S.hist, S.hist, rneed);
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
  uint32_t nw = 0, nt = 0;
#pragma unroll
  for (int i = 0; i < VPT; ++i)
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const uint32_t key = order_key(f4_get(v[i], l));
      const bool valid = (ln[i] >> l) & 1u;
      nw += valid && (ge ? (key & pmask) >= prefix : key > prefix);
      nt += valid && !ge && key == prefix;
    }
  uint32_t ws, ts;
  block_prefix2(nw, nt, ws, ts);
  if ((nw && ws < tie_base) || (nt && ts < nties)) {
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const float e = f4_get(v[i], l);
        const uint32_t key = order_key(e);
        const bool valid = (ln[i] >> l) & 1u;
        const int32_t jw = 4 * (i * T + tid) + l - lead;
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
  if (stats) {
    stats[0] = PATH_SHORT_KERNEL_RADIX;
    stats[1] = int32_t(m);
    stats[2] = 1;
    stats[3] = 0;
  }
}

}  // namespace gvr
