// gvr_kernel.cuh -- the GVR (Guess-Verify-Refine) exact per-row top-K kernel for sm_103a.
//
// One thread-block cluster selects one row.  The row's valid window is split evenly over the
// cluster's CTAs; every CTA holds its share of the row in registers as float4 vectors (read
// from HBM exactly once), so all later passes run over registers.  Per row:
//
//   Guess   uniform block64 sampling: K scores in K/64 runs of 64 consecutive scores whose
//           starts spread evenly over the window, first run at 0, last run ending at nv.
//           GMIN / GMAX are the smallest / largest finite sample ("GVR K=2048 reg_clus with
//           block64 sampling and parallel rescue", TensorRT-LLM PR #20998, "What changes").
//   Verify  a value histogram of NB bins over [GMIN, GMAX] (values above GMAX saturate into
//           the top bin, below GMIN into bin 0); its cluster-wide suffix sums locate the bin
//           b* that crosses the K-th largest value tau ("Why the GLM row overflows").
//   Refine  scores in bins above b* are winners and are written at once; the m members of
//           b* go to a bounded candidate buffer in cluster rank 0, which picks the remaining
//           need = K - above winners exactly.
//   Rescue  an invalid bracket (no finite sample, or GMIN == GMAX) or m above the buffer
//           capacity sends the row to an exact radix select over the 32-bit order-preserving
//           keys of every score, four 8-bit digit passes whose digit histograms are summed
//           over all CTAs of the cluster through distributed shared memory -- the parallel
//           rescue of PR #20998, in the same launch, with no host synchronization.
//
// Two implementation choices keep the per-score work to a compare or two:
//  * sampled histogram floor: the samples also give a floor bin F below which, by the sample
//    quantile, the crossing should not lie; only scores in bins >= F are counted.  A score's
//    bin is >= F exactly when the score is >= v_F, the smallest float whose bin is >= F (found
//    by a 32-way search over float keys), so the floor test is one float compare.  If fewer
//    than K scores reach the floor, the bins below it are counted in a second round, so the
//    result never depends on the floor.
//  * warp-aggregated shared-memory atomics (__match_any_sync) for every histogram update,
//    so tie-heavy rows cost one atomic per distinct bin per warp instruction.
//
// The bin function is monotone non-decreasing in the score (IEEE round-to-nearest subtract and
// multiply by a positive scale, clamp, truncate), which is all the crossing-bin logic needs;
// it is evaluated with the same instruction sequence everywhere, so every pass and every CTA
// classifies a score identically.
#pragma once

#include <cfloat>
#include <cstdint>

#include "gvr_device.cuh"

namespace gvr {

constexpr int NB = 2048;              // value-histogram bins over [GMIN, GMAX]
constexpr int NCOARSE = 256;          // bins of the sample histogram that sets the floor
constexpr int COARSE_SHIFT = 3;       // NB / NCOARSE == 8
constexpr int CAP = 4096;             // candidate slots in cluster rank 0
constexpr int RANK_REFINE_MAX = 256;  // m at or below: refine by pairwise ranking
constexpr int MAX_K = 2048;

enum : int32_t { MODE_DECODE = 0, MODE_PREFILL = 1 };
enum : int32_t { FLAG_FORCE_RESCUE = 1, FLAG_NO_FLOOR = 2, FLAG_ZERO_CAP = 4, FLAG_RADIX_REFINE = 8 };
enum : int32_t {
  PATH_SHORT = 0,
  PATH_REFINE = 1,
  PATH_RESCUE_BRACKET = 2,
  PATH_RESCUE_OVERFLOW = 3,
  PATH_RESCUE_FORCED = 4
};

struct Params {
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
  int32_t flags;
};

struct Crossing {
  int32_t bin;          // b*
  uint32_t above;       // cluster-wide count in bins above b*
  uint32_t m;           // cluster-wide count in b*
  uint32_t base_above;  // count in bins above b* held by lower-ranked CTAs
  uint32_t base_cand;   // count in b* held by lower-ranked CTAs
  uint32_t total;       // cluster-wide count over the bins examined
};

struct alignas(16) Smem {
  uint32_t hist[NB];
  uint32_t dhist[2][256];
  uint32_t shist[NCOARSE];
  float cand_v[CAP];
  int32_t cand_j[CAP];
  uint32_t wsum[2][32];
  float wmin[32];
  float wmax[32];
  Crossing cross;
  float vfloor;
  int32_t floor_bin;
  uint32_t dsel, dabove, dcnt;
  uint32_t ctr_win, ctr_cand;   // this CTA's slot counters (refine path)
  uint32_t ctr_rwin, ctr_rtie;  // rank 0's counters for its own radix refine
  uint32_t rc_win, rc_tie;      // rank 0's counters shared by the cluster in rescue
};

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

// hist[b] += 1 for every lane with pr set, one shared-memory atomic per distinct b per warp.
// Warp-collective.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool pr, uint32_t b) {
  const unsigned act = __ballot_sync(FULL_MASK, pr);
  if (pr) {
    const unsigned peers = __match_any_sync(act, b);
    if ((peers & lanemask_lt()) == 0) atomicAdd(&hist[b], uint32_t(__popc(peers)));
  }
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

// Same, on a counter in another CTA's shared memory (DSMEM address).  Warp-collective.
__device__ __forceinline__ uint32_t warp_alloc_remote(uint32_t ctr_addr, bool want) {
  const unsigned mask = __ballot_sync(FULL_MASK, want);
  uint32_t base = 0;
  if (mask) {
    const int leader = __ffs(mask) - 1;
    if ((threadIdx.x & 31) == leader) base = dsmem_atom_add(ctr_addr, uint32_t(__popc(mask)));
    base = __shfl_sync(FULL_MASK, base, leader);
  }
  return base + __popc(mask & lanemask_lt());
}

// Sum the value histograms of cluster ranks [0, cs) over bins >= fbin and find the crossing
// bin: the highest b with sum_{bins >= b} count >= k.  Thread t owns the NB/T bins
// NB-1-(NB/T)t down to NB-(NB/T)(t+1), so thread order is descending bin order.
template <int T>
__device__ __forceinline__ Crossing reduce_crossing(Smem& S, uint32_t cs, uint32_t rank, uint32_t k,
                                                    int fbin) {
  constexpr int BPT = NB / T;
  constexpr int NW = T / 32;
  static_assert(BPT == 4 || BPT == 8, "threads per CTA must be 256 or 512");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo_bin = NB - BPT * (tid + 1);
  uint32_t tot[BPT], pre[BPT];
#pragma unroll
  for (int j = 0; j < BPT; ++j) tot[j] = pre[j] = 0;
  if (lo_bin + BPT - 1 >= fbin) {
    const uint32_t local = smem_u32(&S.hist[lo_bin]);
    for (uint32_t c = 0; c < cs; ++c) {
      const uint32_t addr = dsmem_map(local, c);
#pragma unroll
      for (int q = 0; q < BPT / 4; ++q) {
        const uint4 v = dsmem_ld_v4(addr + 16u * q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = BPT - 1 - (4 * q + e);  // descending position of bin lo_bin + 4q + e
          tot[j] += w[e];
          if (c < rank) pre[j] += w[e];
        }
      }
    }
  }
  uint32_t st = 0, sp = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    st += tot[j];
    sp += pre[j];
  }
  uint32_t it = st, ip = sp;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(FULL_MASK, it, o);
    const uint32_t b = __shfl_up_sync(FULL_MASK, ip, o);
    if (lane >= o) {
      it += a;
      ip += b;
    }
  }
  if (lane == 31) {
    S.wsum[0][warp] = it;
    S.wsum[1][warp] = ip;
  }
  __syncthreads();
  uint32_t wt = 0, wp = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t x = S.wsum[0][w];
    if (w < warp) {
      wt += x;
      wp += S.wsum[1][w];
    }
    total += x;
  }
  const uint32_t et = wt + it - st;  // count in bins above this thread's bins
  const uint32_t ep = wp + ip - sp;
  if (et < k && et + st >= k) {
    uint32_t cum = et, cp = ep;
#pragma unroll
    for (int j = 0; j < BPT; ++j) {
      if (cum + tot[j] >= k) {
        S.cross.bin = lo_bin + BPT - 1 - j;
        S.cross.above = cum;
        S.cross.m = tot[j];
        S.cross.base_above = cp;
        S.cross.base_cand = pre[j];
        break;
      }
      cum += tot[j];
      cp += pre[j];
    }
  }
  __syncthreads();
  Crossing r = S.cross;
  r.total = total;
  return r;
}

// Sum the 256-bin digit histograms dhist[buf] of cluster ranks [c0, c0 + cn) and find the
// digit d (scanning from 255 down) where the running count reaches `need`; publishes d, the
// count above d and the count at d in S.dsel / S.dabove / S.dcnt.
template <int T>
__device__ __forceinline__ void digit_cross(Smem& S, int buf, uint32_t c0, uint32_t cn, uint32_t need) {
  static_assert(T >= 256, "one thread per digit");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t tot = 0;
  const int d = 255 - tid;
  if (tid < 256) {
    const uint32_t local = smem_u32(&S.dhist[buf][d]);
    for (uint32_t c = c0; c < c0 + cn; ++c) tot += dsmem_ld_u32(dsmem_map(local, c));
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t a = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += a;
  }
  if (lane == 31 && warp < 8) S.wsum[0][warp] = incl;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp && w < 8; ++w) before += S.wsum[0][w];
  const uint32_t excl = before + incl - tot;
  if (tid < 256 && excl < need && excl + tot >= need) {
    S.dsel = uint32_t(d);
    S.dabove = excl;
    S.dcnt = tot;
  }
  __syncthreads();
}

template <int T, int VPT>
__global__ void __launch_bounds__(T, 1024 / T) gvr_topk_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  constexpr int NW = T / 32;
  constexpr int CH = T * VPT;               // vectors per chunk of a CTA's share
  constexpr int KPT = (MAX_K + T - 1) / T;  // samples per thread at most
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t cs = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t row = cluster_id_x();
  const int32_t k = p.k;

  // ---------------------------------------------------------------- row geometry
  // row_stride < 2^31, so window offsets and lengths fit in 32 bits.
  int32_t a = 0, nv = 0;
  if (p.mode == MODE_DECODE) {
    const int64_t kv = p.kv_lens[row / p.next_n];
    int64_t n = 0;
    if (kv >= p.next_n) n = (kv - p.next_n + row % p.next_n + 1) / p.compress_ratio;
    nv = int32_t(n < p.row_stride ? n : p.row_stride);
  } else {
    const int64_t ks = p.row_starts[row];
    const int64_t ke = p.row_ends[row];
    const int64_t s = ks > 0 ? ks : 0;
    const int64_t e = ke < p.row_stride ? ke : p.row_stride;
    a = int32_t(s < p.row_stride ? s : p.row_stride);
    nv = int32_t(e > s ? e - s : 0);
  }
  const float* rowp = p.logits + row * p.row_stride;
  int32_t* out = p.indices + row * int64_t(k);
  float* outv = p.values ? p.values + row * int64_t(k) : nullptr;
  int32_t* stats = (p.row_stats && rank == 0 && tid == 0) ? p.row_stats + 4 * row : nullptr;

  // ---------------------------------------------------------------- short row: identity
  if (nv <= k) {
    for (int i = int(rank) * T + tid; i < k; i += int(cs) * T) {
      out[i] = i < nv ? i : -1;
      if (outv) outv[i] = i < nv ? rowp[a + i] : -FLT_MAX;
    }
    if (stats) {
      stats[0] = PATH_SHORT;
      stats[1] = stats[2] = stats[3] = 0;
    }
    return;
  }

  for (int i = tid; i < NB; i += T) S.hist[i] = 0;
  for (int i = tid; i < NCOARSE; i += T) S.shist[i] = 0;
  if (tid == 0) {
    S.ctr_win = S.ctr_cand = S.ctr_rwin = S.ctr_rtie = 0;
    S.rc_win = S.rc_tie = 0;
    S.cross = Crossing{};
    S.dsel = S.dabove = S.dcnt = 0;
  }

  // ---------------------------------------------------------------- this CTA's share
  // Vectors are 16-byte aligned float4s starting at the aligned column at or below the
  // window start; the first `lead` lanes of vector 0 and the lanes past the window end in the
  // last vector are outside the window and are masked by position.
  const int32_t lead = a & 3;
  const float* base = rowp + (a - lead);
  const int32_t span = lead + nv;
  const int32_t ffull = span >> 2;  // whole vectors inside [col0, window end)
  const int32_t tailn = span & 3;   // in-window scalars of the partial last vector
  const int32_t nvec = ffull + (tailn ? 1 : 0);
  const int32_t per = int32_t((nvec + int32_t(cs) - 1) / int32_t(cs));
  const int32_t vb = int32_t(rank) * per;
  const int32_t ve = vb + per < nvec ? vb + per : nvec;
  const int32_t nchunks = ve > vb ? (ve - vb + CH - 1) / CH : 0;
  const bool resident = nchunks <= 1;

  float4 x[VPT];
  auto vec_index = [&](int ch, int i) -> int32_t { return vb + ch * CH + i * T + tid; };
  auto load_chunk = [&](int ch) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int32_t f = vec_index(ch, i);
      if (f < ve && f < ffull) {
        x[i] = ld_stream_v4(base + 4 * size_t(f));
      } else if (f < ve) {  // the partial last vector: read only its in-window scalars
        const float* q = base + 4 * size_t(f);
        float4 t = f4_zero();
        t.x = q[0];
        if (tailn > 1) t.y = q[1];
        if (tailn > 2) t.z = q[2];
        x[i] = t;
      } else {
        x[i] = f4_zero();
      }
    }
  };
  auto lane_mask = [&](int32_t f) -> uint32_t {
    if (f >= ve) return 0u;
    uint32_t m = 0xFu;
    if (f == 0) m &= (0xFu << lead) & 0xFu;
    if (f == ffull) m &= (1u << tailn) - 1u;
    return m;
  };
  if (nchunks == 1) {
    load_chunk(0);  // stays in registers for every pass
  } else {
#pragma unroll
    for (int i = 0; i < VPT; ++i) x[i] = f4_zero();
  }

  // ---------------------------------------------------------------- guess: block64 sample
  const int nblk = k >> 6;
  float sv[KPT];
  float lmin = INFINITY, lmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int i = q * T + tid;
    sv[q] = __int_as_float(0x7fffffff);
    if (i < k) {
      const int64_t blk = i >> 6;
      const int32_t s = int32_t(blk * (nv - 64) / (nblk - 1));
      const float v = __ldg(rowp + a + s + (i & 63));
      sv[q] = v;
      if (isfinite(v)) {
        lmin = fminf(lmin, v);
        lmax = fmaxf(lmax, v);
      }
    }
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
  gmin = __fadd_rn(gmin, 0.0f);  // -0 -> +0, so every CTA holds the same bits
  const bool bracket_ok = isfinite(gmin) && isfinite(gmax) && gmin < gmax;

  int path = PATH_REFINE;
  if (p.flags & FLAG_FORCE_RESCUE) path = PATH_RESCUE_FORCED;
  else if (!bracket_ok) path = PATH_RESCUE_BRACKET;

  float sc = 0.f;
  float vfloor = -INFINITY;
  int fbin = 0;
  Crossing cr{};
  int rounds = 0;
  if (path == PATH_REFINE) {
    sc = __fdiv_rn(float(NB), __fsub_rn(gmax, gmin));
    // ------------------------------------------------------------ sampled floor
    if (!(p.flags & FLAG_NO_FLOOR)) {
      // about k*k/nv samples are expected above tau; keep twice that plus a margin
      const int64_t want64 = 2 * int64_t(k) * k / nv + 32;
      const uint32_t want = uint32_t(want64 < k ? want64 : k);
#pragma unroll
      for (int q = 0; q < KPT; ++q)
        if (!isnan(sv[q])) atomicAdd(&S.shist[value_bin(sv[q], gmin, sc) >> COARSE_SHIFT], 1u);
      __syncthreads();
      if (warp == 0) {
        uint32_t c[8];
        uint32_t s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = S.shist[NCOARSE - 1 - 8 * lane - i];
          s += c[i];
        }
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += t;
        }
        const uint32_t excl = incl - s;
        const unsigned hm = __ballot_sync(FULL_MASK, excl < want && incl >= want);
        int fc = 0;
        if (hm) {
          const int src = __ffs(hm) - 1;
          if (lane == src) {
            uint32_t cum = excl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              cum += c[i];
              if (cum >= want) {
                fc = NCOARSE - 1 - 8 * lane - i;
                break;
              }
            }
          }
          fc = __shfl_sync(FULL_MASK, fc, src);
        }
        const int fb = fc << COARSE_SHIFT;
        const float vf = fb > 0 ? floor_value(fb, gmin, sc) : -INFINITY;
        if (lane == 0) {
          S.floor_bin = fb;
          S.vfloor = vf;
        }
      }
      __syncthreads();
      fbin = S.floor_bin;
      vfloor = S.vfloor;
    }

    // ------------------------------------------------------------ verify: value histogram
    for (int round = 0; round < 2; ++round) {
      const bool upper = round == 0;
      ++rounds;
      for (int ch = 0; ch < nchunks; ++ch) {
        if (!resident) load_chunk(ch);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const uint32_t m = lane_mask(vec_index(ch, i));
#pragma unroll
          for (int l = 0; l < 4; ++l) {
            const float e = f4_get(x[i], l);
            const bool pr = ((m >> l) & 1u) && (upper ? e >= vfloor : e < vfloor);
            hist_add(S.hist, pr, uint32_t(pr ? value_bin(e, gmin, sc) : 0));
          }
        }
      }
      cluster_sync();
      cr = reduce_crossing<T>(S, cs, rank, uint32_t(k), upper ? fbin : 0);
      if (cr.total >= uint32_t(k)) break;
      if (!upper || fbin == 0) break;  // fewer than k countable scores (NaN in the window)
    }
    const uint32_t cap = (p.flags & FLAG_ZERO_CAP) ? 0u : uint32_t(CAP);
    if (cr.total < uint32_t(k) || cr.m > cap) path = PATH_RESCUE_OVERFLOW;
  }

  if (path == PATH_REFINE) {
    // ------------------------------------------------------------ collect
    const float thr = rounds > 1 ? -INFINITY : vfloor;  // every counted score is >= thr
    const int bstar = cr.bin;
    const uint32_t rv = dsmem_map(smem_u32(&S.cand_v[0]), 0);
    const uint32_t rj = dsmem_map(smem_u32(&S.cand_j[0]), 0);
    for (int ch = 0; ch < nchunks; ++ch) {
      if (!resident) load_chunk(ch);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int32_t f = vec_index(ch, i);
        const uint32_t m = lane_mask(f);
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          const float e = f4_get(x[i], l);
          const bool pr = ((m >> l) & 1u) && e >= thr;
          const int b = pr ? value_bin(e, gmin, sc) : -1;
          const int32_t j = 4 * f + l - lead;
          const uint32_t ws = warp_alloc_local(&S.ctr_win, b > bstar);
          if (b > bstar) {
            const uint32_t slot = cr.base_above + ws;
            if (slot < uint32_t(k)) {  // always true: counts match the histogram's
              out[slot] = j;
              if (outv) outv[slot] = e;
            }
          }
          const uint32_t cslot = warp_alloc_local(&S.ctr_cand, b == bstar);
          if (b == bstar) {
            const uint32_t s = cr.base_cand + cslot;
            if (s < uint32_t(CAP)) {  // always true: m <= CAP on this path
              dsmem_st_u32(rv + 4u * s, __float_as_uint(e));
              dsmem_st_u32(rj + 4u * s, uint32_t(j));
            }
          }
        }
      }
    }
    cluster_sync();  // every candidate has landed in rank 0's buffer
    if (rank != 0) return;

    // ------------------------------------------------------------ refine (rank 0)
    const uint32_t need = uint32_t(k) - cr.above;
    const uint32_t mm = cr.m < uint32_t(CAP) ? cr.m : uint32_t(CAP);
    if (mm <= uint32_t(RANK_REFINE_MAX) && !(p.flags & FLAG_RADIX_REFINE)) {
      // rank of candidate i = number of candidates ordered before it by (value desc, index asc)
      for (uint32_t i = tid; i < mm; i += T) {
        const float v = S.cand_v[i];
        const int32_t j = S.cand_j[i];
        uint32_t r = 0;
        for (uint32_t q = 0; q < mm; ++q) {
          const float w = S.cand_v[q];
          const int32_t jj = S.cand_j[q];
          r += (w > v) || (w == v && jj < j);
        }
        if (r < need && cr.above + r < uint32_t(k)) {
          out[cr.above + r] = j;
          if (outv) outv[cr.above + r] = v;
        }
      }
    } else {
      uint32_t prefix = 0, pmask = 0, rneed = need;
      bool ge = false;
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += T) S.dhist[0][i] = 0;
        __syncthreads();
        for (uint32_t b0 = 0; b0 < mm; b0 += T) {
          const uint32_t i = b0 + tid;
          const bool in = i < mm;
          const uint32_t key = in ? order_key(S.cand_v[i]) : 0u;
          const bool pr = in && (key & pmask) == prefix;
          hist_add(S.dhist[0], pr, (key >> shift) & 255u);
        }
        __syncthreads();
        digit_cross<T>(S, 0, rank, 1, rneed);
        const uint32_t d = S.dsel, ab = S.dabove, cnt = S.dcnt;
        prefix |= d << shift;
        pmask |= 0xFFu << shift;
        rneed -= ab;
        __syncthreads();
        if (cnt == rneed) {
          ge = true;
          break;
        }
      }
      const uint32_t nties = ge ? 0u : rneed;
      const uint32_t win_base = cr.above, tie_base = cr.above + (need - nties);
      for (uint32_t b0 = 0; b0 < mm; b0 += T) {
        const uint32_t i = b0 + tid;
        const bool in = i < mm;
        const uint32_t key = in ? order_key(S.cand_v[i]) : 0u;
        const bool win = in && (ge ? (key & pmask) >= prefix : key > prefix);
        const bool tie = in && !ge && key == prefix;
        const uint32_t ws = warp_alloc_local(&S.ctr_rwin, win);
        if (win && win_base + ws < tie_base) {
          out[win_base + ws] = S.cand_j[i];
          if (outv) outv[win_base + ws] = S.cand_v[i];
        }
        const uint32_t ts = warp_alloc_local(&S.ctr_rtie, tie);
        if (tie && ts < nties) {
          out[tie_base + ts] = S.cand_j[i];
          if (outv) outv[tie_base + ts] = S.cand_v[i];
        }
      }
    }
    if (stats) {
      stats[0] = PATH_REFINE;
      stats[1] = int32_t(cr.m);
      stats[2] = rounds;
      stats[3] = int32_t(cr.above);
    }
    return;
  }

  // ---------------------------------------------------------------- rescue: cluster radix select
  uint32_t prefix = 0, pmask = 0, need = uint32_t(k);
  bool ge = false;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int buf = pass & 1;
    for (int i = tid; i < 256; i += T) S.dhist[buf][i] = 0;
    __syncthreads();
    for (int ch = 0; ch < nchunks; ++ch) {
      if (!resident) load_chunk(ch);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const uint32_t m = lane_mask(vec_index(ch, i));
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          const uint32_t key = order_key(f4_get(x[i], l));
          const bool pr = ((m >> l) & 1u) && (key & pmask) == prefix;
          hist_add(S.dhist[buf], pr, (key >> shift) & 255u);
        }
      }
    }
    cluster_sync();
    digit_cross<T>(S, buf, 0, cs, need);
    const uint32_t d = S.dsel, ab = S.dabove, cnt = S.dcnt;
    prefix |= d << shift;
    pmask |= 0xFFu << shift;
    need -= ab;
    if (cnt == need) {
      ge = true;
      break;
    }
  }
  const uint32_t nties = ge ? 0u : need;
  const uint32_t tie_base = uint32_t(k) - nties;
  const uint32_t rwin = dsmem_map(smem_u32(&S.rc_win), 0);
  const uint32_t rtie = dsmem_map(smem_u32(&S.rc_tie), 0);
  for (int ch = 0; ch < nchunks; ++ch) {
    if (!resident) load_chunk(ch);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int32_t f = vec_index(ch, i);
      const uint32_t m = lane_mask(f);
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const float e = f4_get(x[i], l);
        const uint32_t key = order_key(e);
        const bool valid = (m >> l) & 1u;
        const bool win = valid && (ge ? (key & pmask) >= prefix : key > prefix);
        const bool tie = valid && !ge && key == prefix;
        const int32_t j = 4 * f + l - lead;
        const uint32_t ws = warp_alloc_remote(rwin, win);
        if (win && ws < tie_base) {
          out[ws] = j;
          if (outv) outv[ws] = e;
        }
        const uint32_t ts = warp_alloc_remote(rtie, tie);
        if (tie && ts < nties) {
          out[tie_base + ts] = j;
          if (outv) outv[tie_base + ts] = e;
        }
      }
    }
  }
  cluster_sync();  // rank 0's counters stay alive until every CTA is done with them
  if (stats) {
    stats[0] = path;
    stats[1] = int32_t(cr.m);
    stats[2] = rounds;
    stats[3] = 0;
  }
}

}  // namespace gvr
