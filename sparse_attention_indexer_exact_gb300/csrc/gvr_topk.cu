// gvr_topk.cu -- host side of libgvrtopk: argument validation, launch geometry and the
// C entry points declared in include/gvr_topk.h.
//
// Every entry point checks its arguments on the host, picks a launch geometry from host-known
// quantities only (row stride, row count, k, the device's SM count) and enqueues one
// cluster launch of gvr_topk_kernel on the caller's stream.  Nothing is allocated, no device
// memory is read on the host and nothing synchronizes, so a call costs one launch.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "gvr_kernel.cuh"
#include "gvr_short.cuh"
#include "gvr_split.cuh"
#include "gvr_topk.h"

namespace {

constexpr int kThreads = gvr::THREADS;
constexpr int kMaxDevices = 64;
constexpr int kMaxCluster = 16;  // 16 is a non-portable cluster size (checked per ring depth)
constexpr int64_t kShareVec = 8192;  // largest float4 share per CTA before rows are split further
constexpr int kListTarget = 480;       // expected first-pass list entries per CTA (of LIST_CAP)
constexpr int kListTarget16 = 680;     // the same for the compact lists (of LIST_CAP16)
constexpr int64_t kCheapRereadStages = 4;

struct DeviceState {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int sms = 0;
  int smem_per_sm = 0;     // shared memory per SM (bytes)
  int smem_reserved = 0;   // shared memory the system reserves per CTA (bytes)
  // a 16-CTA cluster can be scheduled at this ring depth: 0 unknown, 1 yes, 2 no (written by any
  // host thread that launches first, so atomic)
  std::atomic<int> fits16[gvr::MAX_STAGES + 1] = {};
};

constexpr int kDefaultSmemPerSm = 228 * 1024;
constexpr int kDefaultSmemReserved = 1024;
constexpr int kMaxCtasPerSm = 7;  // registers: 128 threads x up to 72 registers
DeviceState g_devices[kMaxDevices];

template <int X, bool L16>
cudaError_t set_attributes_of() {
  cudaError_t e = cudaFuncSetAttribute(gvr::gvr_topk_kernel<X, L16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       gvr::smem_bytes(gvr::MAX_STAGES));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gvr::gvr_topk_kernel<X, L16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t set_attributes() {
  cudaError_t e = set_attributes_of<gvr::KX_PLAIN, false>();
  if (e == cudaSuccess) e = set_attributes_of<gvr::KX_EXT, false>();
  if (e == cudaSuccess) e = set_attributes_of<gvr::KX_BLOCKSKIP, false>();
  if (e == cudaSuccess) e = set_attributes_of<gvr::KX_PLAIN, true>();
  if (e == cudaSuccess) e = set_attributes_of<gvr::KX_EXT, true>();
  if (e == cudaSuccess) e = set_attributes_of<gvr::KX_BLOCKSKIP, true>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gvr::gvr_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gvr::split_smem_bytes());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gvr::gvr_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(gvr::short_smem_bytes(gvr::SHORT_MAX)));
  return e;
}

// One-time per-device set-up: kernel attributes, SM count and shared-memory capacity.
cudaError_t device_state(int* sms, int* smem_per_sm, int* smem_reserved) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceState& st = g_devices[dev];
  std::call_once(st.once, [&st, dev]() {
    cudaError_t r = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess)
      r = cudaDeviceGetAttribute(&st.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (r == cudaSuccess)
      r = cudaDeviceGetAttribute(&st.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (r == cudaSuccess) r = set_attributes();
    st.err = r;
  });
  *sms = st.sms;
  *smem_per_sm = st.smem_per_sm;
  *smem_reserved = st.smem_reserved;
  return st.err;
}

bool is_cluster_size(int v) { return v == 1 || v == 2 || v == 4 || v == 8 || v == 16; }

int pow2_ceil(int64_t v) {
  int p = 1;
  while (p < v && p < (1 << 30)) p <<= 1;
  return p;
}

// ws: the *_ws entry points, which also take the flags that choose between the two kernels.
gvr_status check_common(int64_t row_stride, int64_t num_rows, int32_t k, const gvr_options* o, bool ws = false) {
  if (num_rows < 0) return GVR_ERR_ARG;
  if (row_stride < 4 || row_stride % 4 != 0 || row_stride >= (int64_t(1) << 31)) return GVR_ERR_STRIDE;
  if (k != 512 && k != 1024 && k != 2048) return GVR_ERR_K;
  if (o) {
    if (o->reserved != 0) return GVR_ERR_ARG;
    if (o->cluster_size != 0 && !is_cluster_size(o->cluster_size)) return GVR_ERR_ARG;
    if (o->ring_stages != 0 && (o->ring_stages < gvr::MIN_STAGES || o->ring_stages > gvr::MAX_STAGES))
      return GVR_ERR_ARG;
    if (o->flags & ~(GVR_FLAG_FORCE_RESCUE | GVR_FLAG_NO_FLOOR | GVR_FLAG_ZERO_CAP | GVR_FLAG_RADIX_REFINE |
                     GVR_FLAG_DETERMINISTIC | GVR_FLAG_SORTED | GVR_FLAG_STREAM_RESCUE | GVR_FLAG_COMPACT_LISTS |
                     GVR_FLAG_CLUSTER_KERNEL | GVR_FLAG_SPLIT_ALONE | GVR_FLAG_SPLIT_KERNEL |
                     GVR_FLAG_DIAG_FAIL_ROW0 | GVR_FLAG_SHORT_KERNEL | GVR_FLAG_BLOCKSKIP_ALWAYS))
      return GVR_ERR_ARG;
    if (!ws && (o->flags & (GVR_FLAG_SPLIT_ALONE | GVR_FLAG_SPLIT_KERNEL))) return GVR_ERR_ARG;
    if ((o->flags & GVR_FLAG_SHORT_KERNEL) && (o->flags & GVR_FLAG_CLUSTER_KERNEL)) return GVR_ERR_ARG;
  }
  return GVR_OK;
}

// Launch geometry.  Each CTA streams its share of a row through a shared-memory ring, so any
// share length works; the cluster size only balances work.  A row is split so that a CTA's
// share is at most kShareVec float4 (4 CTAs cover a 131072-score row: big batches stay one wave
// of CTAs, whose fixed costs a second wave would repeat); few rows spread each row over more
// CTAs (more SMs pulling one row), down to one ring stage per CTA.
//
// List capacity: the first pass lists every score above the sampled floor, about
// k + 3 sqrt(k nv / s) + 6 nv / s of them for a row of nv scores and s samples (the floor keeps
// mu + 3 sqrt(mu) + 6 samples above it, mu = k s / nv).  A CTA whose list overflows reads its share once
// more, so the row is split at least so finely that a CTA expects to list at most
// kListTarget scores -- unless the share is at most kCheapRereadStages stages, which are
// read again cheaply, or the launch would exceed two waves of CTAs (there the extra CTAs'
// fixed costs outweigh the rereads).
//
// Ring depth: every cluster of the launch should be resident at once (a second wave would
// wait for the whole latency chain of the first), so the ring is as deep as it can be while
// rows x cluster_size CTAs still fit on the GPU, and no deeper than the CTA's share.
struct Geometry {
  int cs;
  int nstage;
  bool l16 = false;  // compact lists (and mu_target 16)
};

int ctas_per_sm(int nstage, int smem_per_sm, int smem_reserved) {
  const int by_smem = smem_per_sm / (gvr::smem_bytes(nstage) + smem_reserved);
  return by_smem < kMaxCtasPerSm ? by_smem : kMaxCtasPerSm;
}

Geometry plan_geometry(int64_t row_stride, int64_t num_rows, int32_t k, int sms, int smem_per_sm,
                       int smem_reserved, const gvr_options* o) {
  const int64_t need_vec = row_stride / 4;
  if (sms <= 0) sms = 148;
  if (smem_per_sm <= 0) smem_per_sm = kDefaultSmemPerSm;
  if (smem_reserved < 0) smem_reserved = kDefaultSmemReserved;
  Geometry g{1, gvr::MIN_STAGES};
  if (o && o->cluster_size) {
    g.cs = o->cluster_size;
  } else {
    int cs_min = pow2_ceil((need_vec + kShareVec - 1) / kShareVec);
    if (cs_min > kMaxCluster) cs_min = kMaxCluster;
    int cs_max = pow2_ceil((need_vec + gvr::STAGE_VEC - 1) / gvr::STAGE_VEC);
    if (cs_max > kMaxCluster) cs_max = kMaxCluster;
    const int64_t slots = int64_t(sms) * ctas_per_sm(gvr::MIN_STAGES, smem_per_sm, smem_reserved);
    const double nv = double(row_stride);
    // scores expected above the sampled floor: (mu + 3 sqrt(mu) + 6) nv / samples, mu = k samples / nv
    const double ns = double(gvr::sample_count(uint32_t(k > 0 ? k : 0), uint32_t(row_stride)));
    const double listed = k > 0 ? double(k) + 3.0 * std::sqrt(double(k) * nv / ns) + 6.0 * nv / ns : 0.0;
    while (cs_min < kMaxCluster && listed > double(kListTarget) * cs_min &&
           (need_vec + int64_t(cs_min) * gvr::STAGE_VEC - 1) / (int64_t(cs_min) * gvr::STAGE_VEC) >
               kCheapRereadStages &&
           num_rows * cs_min * 2 <= 2 * slots)
      cs_min *= 2;
    if (cs_max < cs_min) cs_max = cs_min;
    g.cs = cs_min;
    // widen while the wider launch fills at most half the slots (a quarter for the step to 16,
    // whose CTAs would otherwise share SMs and shallow rings without adding throughput)
    while (g.cs < cs_max && num_rows * g.cs * 2 * (g.cs >= 8 ? 2 : 1) <= slots) g.cs *= 2;
    // Compact lists: when the launch takes two waves of CTAs and half the cluster would fit in
    // one, the 1024-entry lists with 16 samples expected above tau (fewer listed scores) may
    // let half as many CTAs hold each row's list; a second wave would repeat every CTA's
    // fixed latency chain.
    if (g.cs >= 2 && num_rows * g.cs > slots && num_rows * (g.cs / 2) <= slots) {
      const int cs2 = g.cs / 2;
      const double ns16 = double(gvr::sample_count(uint32_t(k > 0 ? k : 0), uint32_t(row_stride), 16u));
      const double listed16 =
          k > 0 ? double(k) + 3.0 * std::sqrt(double(k) * nv / ns16) + 6.0 * nv / ns16 : 0.0;
      const int64_t stages2 = (need_vec + int64_t(cs2) * gvr::STAGE_VEC - 1) / (int64_t(cs2) * gvr::STAGE_VEC);
      if (listed16 <= double(kListTarget16) * cs2 && stages2 <= gvr::LIST_MAX_STAGES) {
        g.cs = cs2;
        g.l16 = true;
      }
    }
  }
  if (o && (o->flags & GVR_FLAG_COMPACT_LISTS)) g.l16 = true;
  if (o && o->ring_stages) {
    g.nstage = o->ring_stages;
  } else {
    const int64_t stages_per_cta = ((need_vec + gvr::STAGE_VEC - 1) / gvr::STAGE_VEC + g.cs - 1) / g.cs;
    const int64_t ctas = num_rows * g.cs;
    const int per_sm_min = ctas_per_sm(gvr::MIN_STAGES, smem_per_sm, smem_reserved);
    for (int d = gvr::MAX_STAGES; d > gvr::MIN_STAGES; --d) {
      if (d > stages_per_cta) continue;
      // a deeper ring that keeps the occupancy of the shallowest one costs nothing; otherwise,
      // as clusters pack into GPCs, leave a tenth of the slots as margin
      const int per_sm = ctas_per_sm(d, smem_per_sm, smem_reserved);
      if (per_sm >= per_sm_min || ctas * 10 <= int64_t(sms) * per_sm * 9) {
        g.nstage = d;
        break;
      }
    }
  }
  return g;
}

// Short-row kernel CTAs resident per SM (1024 threads of at most 32 registers, two by the launch
// bound; fewer when its shared memory does not fit twice) and the waves of them it takes by default.
constexpr int kShortCtasPerSm = 2;
constexpr int kShortWaves = 4;

int64_t short_slots(int64_t row_stride, int sms, int smem_per_sm, int smem_reserved) {
  const int by_smem = smem_per_sm / int(gvr::short_smem_bytes(row_stride) + size_t(smem_reserved));
  return int64_t(sms) * (by_smem < kShortCtasPerSm ? by_smem : kShortCtasPerSm);
}

// The short-row kernel (one CTA per row, the window resident in shared memory) takes the plain
// calls -- no flags, no cluster tuning, not the hinted or block-skip entry points -- whose stride
// fits it and whose rows its CTAs cover in at most kShortWaves waves: measured faster than the
// cluster kernel there (single rows 13-17 %, batches of 16 to 1024 rows 6-35 %), slower on
// batches of thousands of rows (the 4096-row prefill tile), where the cluster kernel streams
// more rows at once.  GVR_FLAG_SHORT_KERNEL (with or without GVR_FLAG_FORCE_RESCUE and
// GVR_FLAG_DIAG_FAIL_ROW0) asks for it whatever the row count; any other flag keeps the cluster
// kernel.
bool use_short(int64_t row_stride, int64_t num_rows, bool plain_entry, int sms, int smem_per_sm,
               int smem_reserved, const gvr_options* o) {
  if (row_stride > gvr::SHORT_MAX || !plain_entry) return false;
  if (o && (o->cluster_size || o->ring_stages)) return false;
  const int32_t flags = o ? o->flags : 0;
  if ((flags & ~(GVR_FLAG_FORCE_RESCUE | GVR_FLAG_DIAG_FAIL_ROW0)) == GVR_FLAG_SHORT_KERNEL) return true;
  if (flags != 0) return false;
  return num_rows <= kShortWaves * short_slots(row_stride, sms, smem_per_sm, smem_reserved);
}

gvr_status launch_short(const gvr::Params& prm, int64_t num_rows, void* stream) {
  if (num_rows > 0x7fffffffLL) return GVR_ERR_ARG;
  gvr::ShortParams q = {};
  q.logits = prm.logits;
  q.row_stride = prm.row_stride;
  q.kv_lens = prm.kv_lens;
  q.row_starts = prm.row_starts;
  q.row_ends = prm.row_ends;
  q.indices = prm.indices;
  q.values = prm.values;
  q.row_stats = prm.row_stats;
  q.next_n = prm.next_n;
  q.compress_ratio = prm.compress_ratio;
  q.k = prm.k;
  q.mode = prm.mode;
  q.flags = prm.flags & (GVR_FLAG_FORCE_RESCUE | GVR_FLAG_DIAG_FAIL_ROW0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(num_rows), 1, 1);
  cfg.blockDim = dim3(gvr::SHORT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = gvr::short_smem_bytes(prm.row_stride);
  cfg.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gvr::gvr_short_kernel, q);
  return e == cudaSuccess ? GVR_OK : GVR_ERR_LAUNCH;
}

gvr_status launch(const gvr::Params& prm, int64_t num_rows, const gvr_options* o, void* stream) {
  int sms = 0, smem_per_sm = 0, smem_reserved = 0;
  if (device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  if (use_short(prm.row_stride, num_rows, !prm.pre_idx && !prm.block_max, sms, smem_per_sm, smem_reserved, o))
    return launch_short(prm, num_rows, stream);
  Geometry geo = plan_geometry(prm.row_stride, num_rows, prm.k, sms, smem_per_sm, smem_reserved, o);
  if (geo.cs == 16 && !(o && o->cluster_size == 16)) {
    // A 16-CTA cluster needs 16 SMs of one GPC with room for it: checked once per ring depth,
    // else the row goes to 8 CTAs.
    int dev = 0;
    cudaGetDevice(&dev);
    std::atomic<int>& fits = g_devices[dev].fits16[geo.nstage];
    int f = fits.load(std::memory_order_relaxed);
    if (f == 0) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(16, 1, 1);
      qc.blockDim = dim3(kThreads, 1, 1);
      qc.dynamicSmemBytes = size_t(gvr::smem_bytes(geo.nstage));
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 16;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.attrs = qa;
      qc.numAttrs = 1;
      int n = 0;
      const cudaError_t qe = cudaOccupancyMaxActiveClusters(&n, gvr::gvr_topk_kernel<gvr::KX_PLAIN, false>, &qc);
      // a refused query leaves its error in the thread's last-error slot: clear that one only
      if (qe != cudaSuccess) cudaGetLastError();
      f = (qe == cudaSuccess && n > 0) ? 1 : 2;
      fits.store(f, std::memory_order_relaxed);
    }
    if (f != 1) {
      gvr_options o8 = o ? *o : gvr_options{};
      o8.cluster_size = 8;
      geo = plan_geometry(prm.row_stride, num_rows, prm.k, sms, smem_per_sm, smem_reserved, &o8);
    }
  }
  const int cs = geo.cs;
  const int64_t blocks = num_rows * cs;
  if (blocks > 0x7fffffffLL) return GVR_ERR_ARG;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = size_t(gvr::smem_bytes(geo.nstage));
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  gvr::Params q = prm;
  q.nstage = geo.nstage;
  q.flags &= ~(GVR_FLAG_CLUSTER_KERNEL | GVR_FLAG_SHORT_KERNEL);
  // the extended instantiation only when a call uses one of its modes; block skipping alone has
  // its own, smaller one
  const int x = ((q.flags & (gvr::FLAG_DETERMINISTIC | gvr::FLAG_SORTED)) || q.pre_idx) ? gvr::KX_EXT
                : q.block_max                                                         ? gvr::KX_BLOCKSKIP
                                                                                      : gvr::KX_PLAIN;
  cudaError_t e;
  if (geo.l16)
    e = x == gvr::KX_EXT         ? cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_EXT, true>, q)
        : x == gvr::KX_BLOCKSKIP ? cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_BLOCKSKIP, true>, q)
                                 : cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_PLAIN, true>, q);
  else
    e = x == gvr::KX_EXT         ? cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_EXT, false>, q)
        : x == gvr::KX_BLOCKSKIP ? cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_BLOCKSKIP, false>, q)
                                 : cudaLaunchKernelEx(&cfg, gvr::gvr_topk_kernel<gvr::KX_PLAIN, false>, q);
  return e == cudaSuccess ? GVR_OK : GVR_ERR_LAUNCH;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ---------------------------------------------------------------- balanced (split) kernel
// Grid: every SM's share of resident CTAs (one chunk each, one wave).  Workspace layout, fixed
// for a device: the per-row arrival counters (SPLIT_MAX_ROWS), the per-chunk counts (grid), the
// published scores and their window indices (grid x SPLIT_UNIT_CAP each).
int64_t split_grid(int sms, int smem_per_sm, int smem_reserved) {
  int per_sm = smem_per_sm / (gvr::split_smem_bytes() + smem_reserved);
  if (per_sm > gvr::SPLIT_CTAS_PER_SM) per_sm = gvr::SPLIT_CTAS_PER_SM;
  if (per_sm < 1) per_sm = 1;
  return int64_t(sms) * per_sm;
}

size_t split_workspace_bytes(int64_t grid) {
  return size_t(gvr::SPLIT_MAX_ROWS) * 4 + size_t(grid) * 4 + size_t(grid) * gvr::SPLIT_UNIT_CAP * 8;
}

constexpr int32_t kSplitFlags = GVR_FLAG_SPLIT_ALONE | GVR_FLAG_SPLIT_KERNEL;

// The balanced kernel for this call, or false when the cluster kernel takes it.
bool use_split(int64_t num_rows, int64_t grid, const gvr_options* o) {
  const int32_t flags = o ? o->flags : 0;
  if (flags & GVR_FLAG_CLUSTER_KERNEL) return false;
  if (flags & ~kSplitFlags) return false;                   // extended modes, cluster diagnostics
  if (o && (o->cluster_size || o->ring_stages)) return false;  // cluster tuning
  if (num_rows > gvr::SPLIT_MAX_ROWS || 2 * num_rows > grid) return false;
  // opt-in: measured slower than the cluster kernel on every workload so far (its fixed chain
  // of schedule, samples, floor, publish and the last CTA's selection is longer)
  return (flags & (GVR_FLAG_SPLIT_KERNEL | GVR_FLAG_SPLIT_ALONE)) != 0;
}

gvr_status launch_split(gvr::SplitParams prm, int64_t grid, void* workspace, void* stream) {
  unsigned char* w = static_cast<unsigned char*>(workspace);
  prm.arrive = reinterpret_cast<uint32_t*>(w);
  prm.surv_n = reinterpret_cast<uint32_t*>(w + size_t(gvr::SPLIT_MAX_ROWS) * 4);
  prm.surv_v = reinterpret_cast<float*>(w + size_t(gvr::SPLIT_MAX_ROWS) * 4 + size_t(grid) * 4);
  prm.surv_j = reinterpret_cast<int32_t*>(w + size_t(gvr::SPLIT_MAX_ROWS) * 4 + size_t(grid) * 4 +
                                          size_t(grid) * gvr::SPLIT_UNIT_CAP * 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = size_t(gvr::split_smem_bytes());
  cfg.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gvr::gvr_split_kernel<true>, prm);
  return e == cudaSuccess ? GVR_OK : GVR_ERR_LAUNCH;
}

// ---------------------------------------------------------------- no-allocation entry point
// topk_decode_noalloc runs the balanced kernel on a scratch area that the library holds as a
// device array of fixed size: its grid is capped at kNoAllocGrid chunks, which fixes the bytes.
constexpr int64_t kNoAllocGrid = 256;
constexpr size_t kNoAllocCounterBytes = size_t(gvr::SPLIT_MAX_ROWS) * 4;
constexpr size_t kNoAllocBytes = kNoAllocCounterBytes + size_t(kNoAllocGrid) * 4 +
                                 size_t(kNoAllocGrid) * gvr::SPLIT_UNIT_CAP * 8;
static_assert(2 * GVR_NOALLOC_MAX_ROWS <= kNoAllocGrid, "the capped grid holds the row limit");
static_assert(int(GVR_FLAG_BLOCKSKIP_ALWAYS) == int(gvr::FLAG_BLOCKSKIP_ALWAYS) &&
                  int(GVR_FLAG_DIAG_FAIL_ROW0) == int(gvr::FLAG_DIAG_FAIL_ROW0),
              "the header's flags are the kernel's");

struct NoAllocState {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  void* scratch = nullptr;  // the device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

}  // namespace

// The scratch itself: every device that loads the library holds these bytes until the process
// exits.  In host code this name is only a host-side stand-in for the device array, so its device
// address is looked up once per device (noalloc_scratch) and that address is what the kernel gets.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

// Device address of the scratch on the current device, looked up on the first call per device
// (with that device current).
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  NoAllocState& st = g_noalloc[dev];
  std::call_once(st.once, [&st]() {
    void* p = nullptr;
    st.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    st.scratch = st.err == cudaSuccess ? p : nullptr;
  });
  *out = st.scratch;
  return st.err;
}

gvr_status check_workspace(void* workspace, size_t bytes, int64_t grid) {
  if (!workspace || !aligned(workspace, 16) || bytes < split_workspace_bytes(grid)) return GVR_ERR_WORKSPACE;
  return GVR_OK;
}

}  // namespace

extern "C" {

gvr_status topk_decode_ex(const float* logits, int64_t row_stride, int64_t num_rows,
                          const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                          int32_t k, int32_t* indices, float* values, void* stream,
                          const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options);
  if (s != GVR_OK) return s;
  if (next_n < 1 || compress_ratio < 1) return GVR_ERR_ARG;
  if (num_rows == 0) return GVR_OK;
  if (!logits || !kv_lens || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(kv_lens, 4) ||
      (values && !aligned(values, 4)))
    return GVR_ERR_ALIGN;
  gvr::Params prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.kv_lens = kv_lens;
  prm.indices = indices;
  prm.values = values;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.next_n = next_n;
  prm.compress_ratio = compress_ratio;
  prm.k = k;
  prm.mode = gvr::MODE_DECODE;
  prm.flags = options ? options->flags : 0;
  return launch(prm, num_rows, options, stream);
}

gvr_status topk_decode_hinted(const float* logits, int64_t row_stride, int64_t num_rows,
                              const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                              int32_t k, const int32_t* pre_idx, int64_t pre_idx_stride,
                              int32_t* indices, float* values, void* stream,
                              const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options);
  if (s != GVR_OK) return s;
  if (next_n < 1 || compress_ratio < 1 || pre_idx_stride < k) return GVR_ERR_ARG;
  if (num_rows == 0) return GVR_OK;
  if (!pre_idx) return GVR_ERR_NULL;
  if (!aligned(pre_idx, 4)) return GVR_ERR_ALIGN;
  // the plain decode checks, then the same launch with hinted sampling
  if (!logits || !kv_lens || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(kv_lens, 4) ||
      (values && !aligned(values, 4)))
    return GVR_ERR_ALIGN;
  gvr::Params prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.kv_lens = kv_lens;
  prm.pre_idx = pre_idx;
  prm.pre_stride = pre_idx_stride;
  prm.indices = indices;
  prm.values = values;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.next_n = next_n;
  prm.compress_ratio = compress_ratio;
  prm.k = k;
  prm.mode = gvr::MODE_DECODE;
  prm.flags = options ? options->flags : 0;
  return launch(prm, num_rows, options, stream);
}

gvr_status topk_decode_blockskip(const float* logits, int64_t row_stride, int64_t num_rows,
                                 const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                                 int32_t k, const float* block_max, int64_t block_max_stride,
                                 int32_t* indices, float* values, void* stream,
                                 const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options);
  if (s != GVR_OK) return s;
  if (next_n < 1 || compress_ratio < 1 || block_max_stride < (row_stride + 31) / 32) return GVR_ERR_ARG;
  if (num_rows == 0) return GVR_OK;
  if (!block_max || !logits || !kv_lens || !indices) return GVR_ERR_NULL;
  if (!aligned(block_max, 4) || !aligned(logits, 16) || !aligned(indices, 4) || !aligned(kv_lens, 4) ||
      (values && !aligned(values, 4)))
    return GVR_ERR_ALIGN;
  gvr::Params prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.kv_lens = kv_lens;
  prm.block_max = block_max;
  prm.bmax_stride = block_max_stride;
  prm.indices = indices;
  prm.values = values;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.next_n = next_n;
  prm.compress_ratio = compress_ratio;
  prm.k = k;
  prm.mode = gvr::MODE_DECODE;
  prm.flags = options ? options->flags : 0;
  return launch(prm, num_rows, options, stream);
}

gvr_status topk_decode(const float* logits, int64_t row_stride, int64_t num_rows,
                       const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio, int32_t k,
                       int32_t* indices, float* values, void* stream) {
  return topk_decode_ex(logits, row_stride, num_rows, kv_lens, next_n, compress_ratio, k, indices,
                        values, stream, nullptr);
}

gvr_status topk_prefill_ex(const float* logits, int64_t row_stride, int64_t num_rows,
                           const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                           int32_t* indices, void* stream, const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options);
  if (s != GVR_OK) return s;
  if (num_rows == 0) return GVR_OK;
  if (!logits || !row_starts || !row_ends || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(row_starts, 4) || !aligned(row_ends, 4))
    return GVR_ERR_ALIGN;
  gvr::Params prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.row_starts = row_starts;
  prm.row_ends = row_ends;
  prm.indices = indices;
  prm.values = nullptr;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.next_n = 1;
  prm.compress_ratio = 1;
  prm.k = k;
  prm.mode = gvr::MODE_PREFILL;
  prm.flags = options ? options->flags : 0;
  return launch(prm, num_rows, options, stream);
}

gvr_status topk_prefill(const float* logits, int64_t row_stride, int64_t num_rows,
                        const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                        int32_t* indices, void* stream) {
  return topk_prefill_ex(logits, row_stride, num_rows, row_starts, row_ends, k, indices, stream, nullptr);
}

const char* gvr_status_string(gvr_status status) {
  switch (status) {
    case GVR_OK: return "ok";
    case GVR_ERR_NULL: return "a required pointer is NULL";
    case GVR_ERR_ALIGN: return "logits must be 16-byte aligned and int32/fp32 buffers 4-byte aligned";
    case GVR_ERR_STRIDE: return "row_stride must be a multiple of 4 in [4, 2^31)";
    case GVR_ERR_K: return "k must be 512, 1024 or 2048";
    case GVR_ERR_ARG: return "invalid argument (row count, next_n, compress_ratio or options)";
    case GVR_ERR_LAUNCH: return "kernel launch failed";
    case GVR_ERR_WORKSPACE: return "workspace is NULL, misaligned or smaller than gvr_workspace_size";
    case GVR_ERR_NOALLOC_LIMIT: return "topk_decode_noalloc takes at most GVR_NOALLOC_MAX_ROWS (128) rows";
  }
  return "unknown status";
}

gvr_status gvr_workspace_size(int32_t sm_count, size_t* bytes) {
  if (!bytes) return GVR_ERR_NULL;
  int sms = sm_count, smem_per_sm = kDefaultSmemPerSm, smem_reserved = kDefaultSmemReserved;
  if (sms <= 0 && device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  *bytes = split_workspace_bytes(split_grid(sms, smem_per_sm, smem_reserved));
  return GVR_OK;
}

gvr_status topk_decode_ws(const float* logits, int64_t row_stride, int64_t num_rows,
                          const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio,
                          int32_t k, int32_t* indices, float* values, void* workspace,
                          size_t workspace_bytes, void* stream, const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options, true);
  if (s != GVR_OK) return s;
  if (next_n < 1 || compress_ratio < 1) return GVR_ERR_ARG;
  if (num_rows == 0) return GVR_OK;
  if (!logits || !kv_lens || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(kv_lens, 4) ||
      (values && !aligned(values, 4)))
    return GVR_ERR_ALIGN;
  int sms = 0, smem_per_sm = 0, smem_reserved = 0;
  if (device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  const int64_t grid = split_grid(sms, smem_per_sm, smem_reserved);
  if (!use_split(num_rows, grid, options)) {
    gvr_options o = options ? *options : gvr_options{};
    o.flags &= ~kSplitFlags;
    return topk_decode_ex(logits, row_stride, num_rows, kv_lens, next_n, compress_ratio, k, indices, values,
                          stream, &o);
  }
  s = check_workspace(workspace, workspace_bytes, grid);
  if (s != GVR_OK) return s;
  gvr::SplitParams prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.kv_lens = kv_lens;
  prm.indices = indices;
  prm.values = values;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.num_rows = int32_t(num_rows);
  prm.next_n = next_n;
  prm.compress_ratio = compress_ratio;
  prm.k = k;
  prm.mode = gvr::MODE_DECODE;
  prm.flags = (options && (options->flags & GVR_FLAG_SPLIT_ALONE)) ? gvr::FLAG_SPLIT_ALONE : 0;
  return launch_split(prm, grid, workspace, stream);
}

gvr_status topk_prefill_ws(const float* logits, int64_t row_stride, int64_t num_rows,
                           const int32_t* row_starts, const int32_t* row_ends, int32_t k,
                           int32_t* indices, void* workspace, size_t workspace_bytes, void* stream,
                           const gvr_options* options) {
  gvr_status s = check_common(row_stride, num_rows, k, options, true);
  if (s != GVR_OK) return s;
  if (num_rows == 0) return GVR_OK;
  if (!logits || !row_starts || !row_ends || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(row_starts, 4) || !aligned(row_ends, 4))
    return GVR_ERR_ALIGN;
  int sms = 0, smem_per_sm = 0, smem_reserved = 0;
  if (device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  const int64_t grid = split_grid(sms, smem_per_sm, smem_reserved);
  if (!use_split(num_rows, grid, options)) {
    gvr_options o = options ? *options : gvr_options{};
    o.flags &= ~kSplitFlags;
    return topk_prefill_ex(logits, row_stride, num_rows, row_starts, row_ends, k, indices, stream, &o);
  }
  s = check_workspace(workspace, workspace_bytes, grid);
  if (s != GVR_OK) return s;
  gvr::SplitParams prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.row_starts = row_starts;
  prm.row_ends = row_ends;
  prm.indices = indices;
  prm.values = nullptr;
  prm.row_stats = options ? options->row_stats : nullptr;
  prm.num_rows = int32_t(num_rows);
  prm.next_n = 1;
  prm.compress_ratio = 1;
  prm.k = k;
  prm.mode = gvr::MODE_PREFILL;
  prm.flags = (options && (options->flags & GVR_FLAG_SPLIT_ALONE)) ? gvr::FLAG_SPLIT_ALONE : 0;
  return launch_split(prm, grid, workspace, stream);
}

gvr_status topk_decode_noalloc(const float* logits, int64_t row_stride, int64_t num_rows,
                               const int32_t* kv_lens, int32_t next_n, int32_t compress_ratio, int32_t k,
                               int32_t* indices, float* values, void* stream) {
  gvr_status s = check_common(row_stride, num_rows, k, nullptr);
  if (s != GVR_OK) return s;
  if (next_n < 1 || compress_ratio < 1) return GVR_ERR_ARG;
  if (num_rows == 0) return GVR_OK;
  if (num_rows > GVR_NOALLOC_MAX_ROWS) return GVR_ERR_NOALLOC_LIMIT;
  if (!logits || !kv_lens || !indices) return GVR_ERR_NULL;
  if (!aligned(logits, 16) || !aligned(indices, 4) || !aligned(kv_lens, 4) ||
      (values && !aligned(values, 4)))
    return GVR_ERR_ALIGN;
  int sms = 0, smem_per_sm = 0, smem_reserved = 0;
  if (device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  int64_t grid = split_grid(sms, smem_per_sm, smem_reserved);
  if (grid > kNoAllocGrid) grid = kNoAllocGrid;
  if (2 * num_rows > grid) return GVR_ERR_NOALLOC_LIMIT;  // a device with fewer SMs than 16
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return GVR_ERR_LAUNCH;
  // The per-row arrival counters must start at zero.  A completed call leaves them so, but the
  // array keeps whatever the last call left (one that was cut short, for instance): clear them.
  if (cudaMemsetAsync(scratch, 0, kNoAllocCounterBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GVR_ERR_LAUNCH;
  gvr::SplitParams prm = {};
  prm.logits = logits;
  prm.row_stride = row_stride;
  prm.kv_lens = kv_lens;
  prm.indices = indices;
  prm.values = values;
  prm.num_rows = int32_t(num_rows);
  prm.next_n = next_n;
  prm.compress_ratio = compress_ratio;
  prm.k = k;
  prm.mode = gvr::MODE_DECODE;
  return launch_split(prm, grid, scratch, stream);
}

gvr_status gvr_plan(int64_t row_stride, int64_t num_rows, int32_t k, const gvr_options* options,
                    int32_t sm_count, int32_t* cluster_size, int32_t* ring_stages, int32_t* threads,
                    int32_t* smem_bytes) {
  gvr_status s = check_common(row_stride, num_rows, k, options);
  if (s != GVR_OK) return s;
  int sms = sm_count, smem_per_sm = kDefaultSmemPerSm, smem_reserved = kDefaultSmemReserved;
  if (sms <= 0 && device_state(&sms, &smem_per_sm, &smem_reserved) != cudaSuccess) return GVR_ERR_LAUNCH;
  if (use_short(row_stride, num_rows, true, sms, smem_per_sm, smem_reserved, options)) {
    if (cluster_size) *cluster_size = 1;
    if (ring_stages) *ring_stages = 0;
    if (threads) *threads = gvr::SHORT_THREADS;
    if (smem_bytes) *smem_bytes = int32_t(gvr::short_smem_bytes(row_stride));
    return GVR_OK;
  }
  const Geometry geo = plan_geometry(row_stride, num_rows, k, sms, smem_per_sm, smem_reserved, options);
  if (cluster_size) *cluster_size = geo.cs;
  if (ring_stages) *ring_stages = geo.nstage;
  if (threads) *threads = kThreads;
  if (smem_bytes) *smem_bytes = int32_t(gvr::smem_bytes(geo.nstage));
  return GVR_OK;
}

}  // extern "C"
