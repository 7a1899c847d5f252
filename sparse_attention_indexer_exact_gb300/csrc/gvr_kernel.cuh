// gvr_kernel.cuh -- the GVR (Guess-Verify-Refine) exact per-row top-K kernel for sm_103a.
//
// One thread-block cluster selects one row.  The row's valid window is split evenly over the
// cluster's CTAs; each CTA stages its share in shared memory with bulk asynchronous copies
// (TMA, completion on an mbarrier), so the row is read from HBM exactly once and every later
// pass reads shared memory.  Per row:
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
// Implementation choices that keep the per-score work to about one compare:
//  * sampled histogram floor: the samples also give a floor bin F below which, by the sample
//    quantile, the crossing should not lie; only scores in bins >= F are counted.  A score's
//    bin is >= F exactly when the score is >= v_F, the smallest float whose bin is >= F (found
//    by a 32-way search over float keys), so the floor test is one float compare.  If fewer
//    than K scores reach the floor, the bins below it are counted in a second round, so the
//    result never depends on the floor.
//  * above-floor bitmask: each thread compares its (at most 32) staged scores with v_F once
//    and keeps a 32-bit mask of the few that pass; the histogram and the collect step then
//    visit only the set bits, reading those scores back from shared memory.  A warp whose
//    masks are dense (tie-heavy rows) counts with warp-aggregated atomics (__match_any_sync)
//    instead, one shared-memory atomic per distinct bin per warp instruction.
//
// The bin function is monotone non-decreasing in the score (IEEE round-to-nearest subtract and
// multiply by a positive scale, clamp, truncate), which is all the crossing-bin logic needs;
// it is evaluated with the same instruction sequence everywhere, so every pass and every CTA
// classifies a score identically.  Positions outside the window (the lead lanes below an
// unaligned window start, the lanes past its end) are never compared: they are staged as NaN,
// which fails every `>=` / `<` test, and the key-space rescue masks them by position.
#pragma once

#include <cfloat>
#include <cstddef>
#include <cstdint>

#include "gvr_device.cuh"

namespace gvr {

constexpr int NB = 2048;              // value-histogram bins over [GMIN, GMAX]
constexpr int NCOARSE = 256;          // bins of the sample histogram that sets the floor
constexpr int COARSE_SHIFT = 3;       // NB / NCOARSE == 8
constexpr int CAP = 4096;             // candidate slots in cluster rank 0
constexpr int RANK_REFINE_MAX = 256;  // m at or below: refine by pairwise ranking
constexpr int MAX_K = 2048;
constexpr int MAX_VPT = 8;            // staged float4 per thread per chunk: a 32-bit score mask
constexpr int SPARSE_MAX = 8;         // above-floor scores per thread beyond which a warp goes dense
constexpr uint32_t COPY_PIECE = 16384;             // bytes per bulk copy instruction
constexpr uint64_t WAIT_LIMIT_NS = 500000000ull;   // bound on any wait for staged data (0.5 s)

enum : int32_t { MODE_DECODE = 0, MODE_PREFILL = 1 };
enum : int32_t { FLAG_FORCE_RESCUE = 1, FLAG_NO_FLOOR = 2, FLAG_ZERO_CAP = 4, FLAG_RADIX_REFINE = 8 };
enum : int32_t {
  PATH_DEVICE_ERROR = -1,
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
  int32_t slice_vec;          // float4 slots of the shared-memory stage per CTA (T * vpt)
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
  uint32_t hist[NB];  // first: 16-byte aligned groups of 4 bins are read as one vector
  uint32_t dhist[2][256];
  uint32_t shist[NCOARSE];
  float cand_v[CAP];
  int32_t cand_j[CAP];
  uint32_t wsum[2][32];
  float wmin[32];
  float wmax[32];
  Crossing cross;
  float vthr;
  int32_t floor_bin;
  uint32_t dsel, dabove, dcnt;
  uint32_t ctr_win, ctr_cand;   // this CTA's slot counters (refine path)
  uint32_t ctr_rwin, ctr_rtie;  // rank 0's counters for its own radix refine
  uint32_t rc_win, rc_tie;      // rank 0's counters shared by the cluster in rescue
  uint32_t tout;                // this CTA gave up waiting for staged data
  uint32_t err;                 // rank 0: some CTA of the cluster gave up
  uint64_t bar;                 // completion of the bulk copies of the current stage
};
static_assert(offsetof(Smem, hist) % 16 == 0, "histogram groups are read as 16-byte vectors");
static_assert(offsetof(Smem, bar) % 8 == 0, "mbarrier must be 8-byte aligned");

constexpr int SMEM_FIXED = int((sizeof(Smem) + 127) / 128 * 128);

__host__ __device__ constexpr int smem_bytes(int slice_vec) { return SMEM_FIXED + 16 * slice_vec; }

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

template <int T>
__global__ void __launch_bounds__(T, 2) gvr_topk_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  float4* sdata = reinterpret_cast<float4*>(smem_raw + SMEM_FIXED);
  const float* sdataf = reinterpret_cast<const float*>(smem_raw + SMEM_FIXED);
  constexpr int NW = T / 32;
  constexpr int KPT = (MAX_K + T - 1) / T;  // samples per thread at most
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t cs = cluster_size();
  const uint32_t rank = cluster_rank();
  const int64_t row = cluster_id_x();
  const int32_t k = p.k;
  const float qnan = __int_as_float(0x7fffffff);

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
    S.tout = S.err = 0;
    S.cross = Crossing{};
    S.dsel = S.dabove = S.dcnt = 0;
    mbar_init(&S.bar, 1);
    mbar_init_fence();
  }

  // ---------------------------------------------------------------- this CTA's share
  // Vectors are 16-byte aligned float4s starting at the aligned column at or below the
  // window start.  The share [vb, ve) is staged in chunks of slice_vec vectors; with one chunk
  // (the usual case) it is staged once and stays resident for every pass.
  const int32_t lead = a & 3;
  const float* base = rowp + (a - lead);
  const int32_t span = lead + nv;
  const int32_t ffull = span >> 2;  // whole vectors inside [col0, window end)
  const int32_t tailn = span & 3;   // in-window scalars of the partial last vector
  const int32_t nvec = ffull + (tailn ? 1 : 0);
  const int32_t per = int32_t((nvec + int32_t(cs) - 1) / int32_t(cs));
  const int32_t vb = int32_t(rank) * per < nvec ? int32_t(rank) * per : nvec;
  const int32_t ve = vb + per < nvec ? vb + per : nvec;
  const int32_t cap_vec = p.slice_vec;
  const int32_t nloc = ve - vb;
  const int nchunks = nloc > 0 ? (nloc + cap_vec - 1) / cap_vec : 0;
  const bool resident = nchunks <= 1;
  uint32_t phase = 0;

  auto chunk_begin = [&](int ch) -> int32_t { return vb + ch * cap_vec; };
  auto chunk_count = [&](int ch) -> int32_t {
    const int32_t c0 = vb + ch * cap_vec;
    return (c0 + cap_vec < ve ? c0 + cap_vec : ve) - c0;
  };
  // Stage chunk ch: bulk copies of its whole vectors (thread 0) and the in-window scalars of
  // the partial last vector.  Returns whether bulk copies were issued (same on all threads).
  auto issue_chunk = [&](int ch) -> bool {
    const int32_t c0 = chunk_begin(ch), c1 = c0 + chunk_count(ch);
    const int32_t fe = c1 < ffull ? c1 : ffull;
    const int32_t nfull = fe > c0 ? fe - c0 : 0;
    if (tid == 0 && nfull > 0) {
      fence_proxy_async_smem();
      const uint32_t bytes = uint32_t(nfull) * 16u;
      mbar_arrive_expect_tx(&S.bar, bytes);
      const char* src = reinterpret_cast<const char*>(base + 4 * size_t(c0));
      char* dst = reinterpret_cast<char*>(sdata);
      for (uint32_t off = 0; off < bytes; off += COPY_PIECE) {
        const uint32_t n = bytes - off < COPY_PIECE ? bytes - off : COPY_PIECE;
        bulk_copy_g2s(dst + off, src + off, n, &S.bar);
      }
    }
    if (tid == 32 && tailn && ffull >= c0 && ffull < c1) {
      const float* q = base + 4 * size_t(ffull);
      sdata[ffull - c0] = make_float4(q[0], tailn > 1 ? q[1] : qnan, tailn > 2 ? q[2] : qnan, qnan);
    }
    return nfull > 0;
  };
  // Wait (bounded) for chunk ch, blank the lead lanes below the window start, publish.
  auto wait_chunk = [&](int ch, bool armed) {
    bool late = false;
    if (armed) {
      if (!mbar_wait_bounded(&S.bar, phase, WAIT_LIMIT_NS)) {
        mbar_wait_bounded(&S.bar, phase, WAIT_LIMIT_NS);  // let copies in flight land
        late = true;
      }
      phase ^= 1u;
    }
    if (tid == 0 && lead > 0 && chunk_begin(ch) == 0 && chunk_count(ch) > 0) {
      float* v0 = reinterpret_cast<float*>(sdata);
      for (int l = 0; l < lead; ++l) v0[l] = qnan;
    }
    if (__syncthreads_or(late) && tid == 0) S.tout = 1;
  };
  // After a cluster barrier: tell rank 0 that this CTA gave up waiting (rank 0 marks the row).
  auto report_timeout = [&]() {
    if (tid == 0 && S.tout) dsmem_st_u32(dsmem_map(smem_u32(&S.err), 0), 1u);
  };
  // Mask of this thread's staged scores that are >= thr (below == false) or < thr (below ==
  // true); bit 4i+l is lane l of the thread's i-th vector (chunk vector i*T + tid).
  auto build_bits = [&](int32_t cnt, float thr, bool below) -> uint32_t {
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < MAX_VPT; ++i) {
      const int32_t f = i * T + tid;
      if (f < cnt) {
        const float4 v = sdata[f];
        uint32_t b;
        if (!below)
          b = uint32_t(v.x >= thr) | (uint32_t(v.y >= thr) << 1) | (uint32_t(v.z >= thr) << 2) |
              (uint32_t(v.w >= thr) << 3);
        else
          b = uint32_t(v.x < thr) | (uint32_t(v.y < thr) << 1) | (uint32_t(v.z < thr) << 2) |
              (uint32_t(v.w < thr) << 3);
        bits |= b << (4 * i);
      }
    }
    return bits;
  };
  auto bit_score = [&](int j) -> float { return sdataf[4 * ((j >> 2) * T + tid) + (j & 3)]; };

  bool armed0 = false;
  if (nchunks == 1) armed0 = issue_chunk(0);  // overlaps the sampling below

  // ---------------------------------------------------------------- guess: block64 sample
  const int nblk = k >> 6;
  float sv[KPT];
  float lmin = INFINITY, lmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int i = q * T + tid;
    sv[q] = qnan;
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
  if (path == PATH_REFINE) {
    sc = __fdiv_rn(float(NB), __fsub_rn(gmax, gmin));
    // ------------------------------------------------------------ sampled floor
    if (!(p.flags & FLAG_NO_FLOOR)) {
      // mu = k*k/nv samples are expected above tau; keep mu + 3 sqrt(mu) + 16 above the floor
      const float mu = float(k) * float(k) / float(nv);
      const float want_f = mu + 3.0f * sqrtf(mu) + 16.0f;
      const uint32_t want = want_f < float(k) ? uint32_t(want_f) : uint32_t(k);
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
          S.vthr = vf;
        }
      }
      __syncthreads();
      fbin = S.floor_bin;
      vfloor = S.vthr;
    }
  }

  if (nchunks == 1) wait_chunk(0, armed0);

  Crossing cr{};
  int rounds = 0;
  uint32_t mbits = 0;  // resident share: this thread's scores >= vfloor
  if (path == PATH_REFINE) {
    // ------------------------------------------------------------ verify: value histogram
    auto count_bits = [&](uint32_t bits) {
      const bool dense = __any_sync(FULL_MASK, __popc(bits) > SPARSE_MAX);
      if (!dense) {
        while (bits) {
          const int j = __ffs(bits) - 1;
          bits &= bits - 1;
          atomicAdd(&S.hist[value_bin(bit_score(j), gmin, sc)], 1u);
        }
      } else {
#pragma unroll 4
        for (int j = 0; j < 4 * MAX_VPT; ++j) {
          const bool pr = (bits >> j) & 1u;
          const float e = pr ? bit_score(j) : 0.f;
          hist_add(S.hist, pr, pr ? uint32_t(value_bin(e, gmin, sc)) : 0u);
        }
      }
    };
    for (int round = 0; round < 2; ++round) {
      const bool upper = round == 0;
      ++rounds;
      if (resident) {
        if (nchunks == 1) {
          const uint32_t b = build_bits(nloc, vfloor, !upper);
          if (upper) mbits = b;
          count_bits(b);
        }
      } else {
        for (int ch = 0; ch < nchunks; ++ch) {
          const bool armed = issue_chunk(ch);
          wait_chunk(ch, armed);
          count_bits(build_bits(chunk_count(ch), vfloor, !upper));
          __syncthreads();
        }
      }
      cluster_sync();
      report_timeout();
      cr = reduce_crossing<T>(S, cs, rank, uint32_t(k), upper ? fbin : 0);
      if (cr.total >= uint32_t(k)) break;
      if (!upper || fbin == 0) break;  // fewer than k countable scores (NaN in the window)
    }
    const uint32_t cap = (p.flags & FLAG_ZERO_CAP) ? 0u : uint32_t(CAP);
    if (cr.total < uint32_t(k) || cr.m > cap) path = PATH_RESCUE_OVERFLOW;
  }

  if (path == PATH_REFINE) {
    // ------------------------------------------------------------ collect
    const int bstar = cr.bin;
    float thr = vfloor;
    if (rounds > 1) {  // scores below the floor were counted too: select bins >= b* afresh
      if (warp == 0) {
        const float t = bstar > 0 ? floor_value(bstar, gmin, sc) : -INFINITY;
        if (lane == 0) S.vthr = t;
      }
      __syncthreads();
      thr = S.vthr;
    }
    const uint32_t rv = dsmem_map(smem_u32(&S.cand_v[0]), 0);
    const uint32_t rj = dsmem_map(smem_u32(&S.cand_j[0]), 0);
    auto collect_bits = [&](uint32_t bits, int32_t c0) {
      while (bits) {
        const int j = __ffs(bits) - 1;
        bits &= bits - 1;
        const float e = bit_score(j);
        const int b = value_bin(e, gmin, sc);
        const int32_t jw = 4 * (c0 + (j >> 2) * T + tid) + (j & 3) - lead;
        if (b > bstar) {
          const uint32_t slot = cr.base_above + atomicAdd(&S.ctr_win, 1u);
          if (slot < uint32_t(k)) {  // always true: counts match the histogram's
            out[slot] = jw;
            if (outv) outv[slot] = e;
          }
        } else if (b == bstar) {
          const uint32_t c = cr.base_cand + atomicAdd(&S.ctr_cand, 1u);
          if (c < uint32_t(CAP)) {  // always true: m <= CAP on this path
            dsmem_st_u32(rv + 4u * c, __float_as_uint(e));
            dsmem_st_u32(rj + 4u * c, uint32_t(jw));
          }
        }
      }
    };
    if (resident) {
      if (nchunks == 1) collect_bits(rounds > 1 ? build_bits(nloc, thr, false) : mbits, vb);
    } else {
      for (int ch = 0; ch < nchunks; ++ch) {
        const bool armed = issue_chunk(ch);
        wait_chunk(ch, armed);
        collect_bits(build_bits(chunk_count(ch), thr, false), chunk_begin(ch));
        __syncthreads();
      }
      report_timeout();
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
    __syncthreads();
    const bool failed = S.err || S.tout;
    if (failed)
      for (int i = tid; i < k; i += T) out[i] = -2;
    if (stats) {
      stats[0] = failed ? PATH_DEVICE_ERROR : PATH_REFINE;
      stats[1] = int32_t(cr.m);
      stats[2] = rounds;
      stats[3] = int32_t(cr.above);
    }
    return;
  }

  // ---------------------------------------------------------------- rescue: cluster radix select
  // Every staged score of the window takes part; positions outside the window are masked here
  // by position (their staged NaN would otherwise have a key).
  auto key_pass = [&](auto&& visit) {
    for (int ch = 0; ch < nchunks; ++ch) {
      if (!resident) {
        const bool armed = issue_chunk(ch);
        wait_chunk(ch, armed);
      }
      const int32_t c0 = chunk_begin(ch), cnt = chunk_count(ch);
#pragma unroll 1
      for (int i = 0; i < MAX_VPT; ++i) {
        const int32_t f = i * T + tid;
        const bool in = f < cnt;
        const float4 v = in ? sdata[f] : f4_zero();
        const int32_t g = c0 + f;  // vector index from the aligned window base
#pragma unroll
        for (int l = 0; l < 4; ++l) {
          const bool valid = in && (g != 0 || l >= lead) && (g != ffull || l < tailn);
          visit(f4_get(v, l), valid, 4 * g + l - lead);
        }
      }
      if (!resident) __syncthreads();
    }
  };
  uint32_t prefix = 0, pmask = 0, need = uint32_t(k);
  bool ge = false;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int buf = pass & 1;
    for (int i = tid; i < 256; i += T) S.dhist[buf][i] = 0;
    __syncthreads();
    key_pass([&](float e, bool valid, int32_t) {
      const uint32_t key = order_key(e);
      const bool pr = valid && (key & pmask) == prefix;
      hist_add(S.dhist[buf], pr, (key >> shift) & 255u);
    });
    cluster_sync();
    report_timeout();
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
  key_pass([&](float e, bool valid, int32_t jw) {
    const uint32_t key = order_key(e);
    const bool win = valid && (ge ? (key & pmask) >= prefix : key > prefix);
    const bool tie = valid && !ge && key == prefix;
    const uint32_t ws = warp_alloc_remote(rwin, win);
    if (win && ws < tie_base) {
      out[ws] = jw;
      if (outv) outv[ws] = e;
    }
    const uint32_t ts = warp_alloc_remote(rtie, tie);
    if (tie && ts < nties) {
      out[tie_base + ts] = jw;
      if (outv) outv[tie_base + ts] = e;
    }
  });
  report_timeout();
  cluster_sync();  // rank 0's counters stay alive until every CTA is done with them
  if (rank == 0) {
    const bool failed = S.err || S.tout;
    if (failed)
      for (int i = tid; i < k; i += T) out[i] = -2;
    if (stats) {
      stats[0] = failed ? PATH_DEVICE_ERROR : path;
      stats[1] = int32_t(cr.m);
      stats[2] = rounds;
      stats[3] = 0;
    }
  }
}

}  // namespace gvr
