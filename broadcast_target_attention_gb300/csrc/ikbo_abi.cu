// C ABI of the IKBO target-attention library: host-side checks, scratch
// space, tensor-map templates and kernel launches.  See include/ikbo.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/ikbo.h"
#include "ikbo_attn_simt.cuh"
#include "ikbo_attn_ab.cuh"
#include "ikbo_attn_pp.cuh"
#include "ikbo_attn_tc.cuh"
#include "ikbo_broadcast.cuh"
#include "ikbo_lce.cuh"
#include "ikbo_common.cuh"
#include "ikbo_plan.cuh"

namespace ikbo {

// Error words (bits kErrIndex, kErrOffsets, kErrTimeout), one per stream:
// word i > 0 belongs to the i-th stream of the device that made a call, in
// order of first use; word 0 is shared by the streams past kErrSlots - 1.
constexpr int kErrSlots = 64;
__device__ int g_ikbo_error_word[kErrSlots];

namespace {

constexpr int kVersion = 10000;  // 1.0.0
constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s bound on any in-kernel wait

struct DeviceState {
  bool ready = false;
  int num_sms = 0;
  int tc_grid[2] = {0, 0};   // CTAs of the tcgen05 kernel (clusters of 2), D = 64 / 128
  int pp_grid[2] = {0, 0};   // CTAs of the two-tile tcgen05 kernel, D = 64 / 128
  int ab_grid[2] = {0, 0};   // CTAs of the key-interleaved tcgen05 kernel, D = 64 / 128
  std::atomic<uint64_t>* calls = nullptr;   // calls so far: the key-interleaved kernel's marker
  bool lce_ready[2][4] = {};      // shared-memory attribute set: by CTA-pair form, N = 64 .. 256
  int lce_clusters[2][4][9] = {};   // co-resident clusters of the LCE kernel, by form, N / 64 and cluster size
  int* err_host = nullptr;       // pinned copy of the error word, made by the host-buffer entry point
  std::mutex* host_call = nullptr;   // serialises that entry point's use of err_host
  // The library's own stream-ordered pool on this device, made by the first
  // call that allocates: it keeps freed scratch between calls (the device's
  // default pool, which other code may use, is left as it is).
  cudaMemPool_t pool = nullptr;
  int* err_word = nullptr;                       // the device's g_ikbo_error_word
  cudaStream_t err_stream[kErrSlots] = {};       // stream of each word (1 .. err_streams)
  int err_streams = 0;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  bool ev_ready = false;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
bool g_timing = false;
int g_timing_dev = -1;
int g_debug_flags = 0;
uint64_t* g_trace = nullptr;
uint64_t g_timeout_ns = kDefaultTimeoutNs;
// Kernel choice of this thread (ikbo_set_kernel): 0 = automatic, 1 = SIMT,
// 2 = tcgen05 with one query tile per item, 3 = tcgen05 with two, 4 =
// tcgen05 with the key tiles of one query tile over two warpgroups.
thread_local int t_kernel = 0;
enum { kKernAuto = 0, kKernSimt = 1, kKernTc = 2, kKernPp = 3, kKernAb = 4 };

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  (void)e;
  return IKBO_ERR_CUDA;
}

// Current device's state, initialised on first use.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IKBO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return IKBO_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return IKBO_ERR_CUDA;
    if (major != 10 || minor != 3) return IKBO_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ikbo_error_word) != cudaSuccess) return IKBO_ERR_CUDA;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return IKBO_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    s.host_call = new std::mutex();   // lives as long as the process, like this state
    s.calls = new std::atomic<uint64_t>(0);
    s.num_sms = sms;
    s.err_word = static_cast<int*>(p);
    s.ready = true;
  }
  *out = &s;
  return IKBO_OK;
}

// The error word of stream `st`: the stream's own once it has one, a new one
// on its first call, the shared word 0 once all are taken.  (A call captured
// in a graph records into the word of the stream it was captured on.)
int error_slot(DeviceState* ds, cudaStream_t st, bool take) {
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int i = 1; i <= ds->err_streams; ++i)
    if (ds->err_stream[i] == st) return i;
  if (!take || ds->err_streams + 1 >= kErrSlots) return 0;
  ds->err_stream[++ds->err_streams] = st;
  return ds->err_streams;
}

int* error_word(DeviceState* ds, cudaStream_t st) { return ds->err_word + error_slot(ds, st, true); }

// `bytes` of scratch from the library's pool on the current device, in
// stream order on `st` (made on first use; freed memory stays in the pool).
// Under stream capture the allocation becomes a graph memory node.
cudaError_t pool_alloc(DeviceState* ds, void** ptr, size_t bytes, cudaStream_t st) {
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!ds->pool) {
      int dev = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e != cudaSuccess) return e;
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.handleTypes = cudaMemHandleTypeNone;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t made = nullptr;
      if ((e = cudaMemPoolCreate(&made, &props)) != cudaSuccess) return e;
      uint64_t keep = UINT64_MAX;
      if ((e = cudaMemPoolSetAttribute(made, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
        cudaMemPoolDestroy(made);
        return e;
      }
      ds->pool = made;
    }
    pool = ds->pool;
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

template <typename T>
cudaError_t pool_alloc(DeviceState* ds, T** ptr, size_t bytes, cudaStream_t st) {
  return pool_alloc(ds, reinterpret_cast<void**>(ptr), bytes, st);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_args(const void* q, const void* k, const void* v, const int32_t* off, const int32_t* c2u,
               int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D, float scale,
               const void* out) {
  if (n_cand < 0 || n_user < 0 || H < 1 || Lq < 1 || Lq > kTileM || (D != 64 && D != 128))
    return IKBO_ERR_SHAPE;
  if (n_cand >= (int64_t(1) << 31) || n_user >= (int64_t(1) << 31) - 1) return IKBO_ERR_SHAPE;
  if (!std::isfinite(scale)) return IKBO_ERR_SCALE;
  if (n_cand == 0) return IKBO_OK;
  if (!q || !k || !v || !off || !c2u || !out) return IKBO_ERR_NULL;
  if (n_user == 0) return IKBO_ERR_INDEX;  // every candidate would point outside [0, 0)
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(off) & 3u) || (reinterpret_cast<uintptr_t>(c2u) & 3u))
    return IKBO_ERR_ALIGN;
  const uintptr_t ob = reinterpret_cast<uintptr_t>(out);
  const uintptr_t oe = ob + uintptr_t(n_cand) * H * Lq * D * 2;
  const uintptr_t qb = reinterpret_cast<uintptr_t>(q);
  const uintptr_t qe = qb + uintptr_t(n_cand) * H * Lq * D * 2;
  if (ob < qe && qb < oe) return IKBO_ERR_ALIAS;
  const uintptr_t kb = reinterpret_cast<uintptr_t>(k), vb = reinterpret_cast<uintptr_t>(v);
  if ((kb >= ob && kb < oe) || (vb >= ob && vb < oe)) return IKBO_ERR_ALIAS;
  return IKBO_OK;
}

// Candidates per query tile: floor(128 / Lq).  The sorted-order Q map's box
// holds a whole tile, so one TMA copy per 64-column block loads a tile (rows
// past the tile's own candidates belong to the next ones, or are zero-filled
// past the end of q; they are never used or stored).
int cands_per_tile(int Lq) { return kTileM / Lq; }
int qbox_cands(int Lq) { return cands_per_tile(Lq); }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Layout of the per-call scratch space.
struct Workspace {
  size_t header, kmap, vmap, items, units, perm, cand_start, scratch, partial_o, partial_ml,
      cta_items, map_slots, item_user, ab_o, ab_lse, ab_flags, clc_slots, total;
  int max_items, max_split_items, max_units, max_cta_items, grid, map_stride;
  int clc_slot_bytes, clc_map_offset;
  int kernel;   // kKernSimt, kKernTc or kKernPp
  bool fused;
  bool clc;     // two-tile kernel with Cluster Launch Control (grid = a bound on the units)
};

// Target-only calls on the two-tile kernel with at most this many users run
// with Cluster Launch Control: one CTA per unit of work (the grid a bound on
// their number), CTAs that finish early taking over those not yet started;
// each SM keeps a slot of the plan's user tables and one bounded V map per user.
constexpr int64_t kClcMaxUsers = 256;

// The grid of the two-tile kernel with Cluster Launch Control: at least one CTA
// per unit (H x two-tile groups of candidates of every user).
int64_t pp_units_bound(int64_t n_cand, int64_t n_user, int H, int Lq) {
  const int64_t pair = 2 * cands_per_tile(Lq);
  return int64_t(H) * ((n_cand + pair - 1) / pair + (n_user < n_cand ? n_user : n_cand));
}

bool fits_in_kernel_planning(int64_t n_cand, int64_t n_user) {
  return n_cand <= kFusedMaxCand && n_user <= kFusedMaxUser;
}

// The automatic choice takes the two-tile kernel when the users have on
// average at least two query tiles each and the batch makes at least this
// many two-tile items (about four per SM of a GB300).  Measured on one GB300
// it is 3-19 % faster than the one-tile kernel on such batches (2 to 64
// tiles per user, 1024 to 4096 items).
constexpr int64_t kPpMinItems = 600;
// ... or at least this many where it deals by Cluster Launch Control and asks
// for each next unit only once the current one's loads are issued (target
// attention alone, at most kClcMaxUsers users, D = 128): there it is 6 %
// faster than the one-tile kernel on ~260 items of very unequal cost
// (Zipf-distributed candidates, 64 to 4096 keys); the two are even on 160
// items of one user.
constexpr int64_t kPpMinItemsClc = 200;

// The kernel the thread's choice gives.  The two-tile and the key-interleaved
// kernels plan in-kernel only, so inputs beyond those limits take the
// one-tile kernel.  target_only: not a fused self + target call.
int kernel_choice(int64_t n_cand, int64_t n_user, int H, int Lq, int D, bool target_only) {
  if (t_kernel == kKernSimt) return kKernSimt;
  if (t_kernel == kKernTc || !fits_in_kernel_planning(n_cand, n_user)) return kKernTc;
  if (t_kernel == kKernPp) return kKernPp;
  // the key-interleaved kernel only when chosen: it is faster when a few
  // units are very long, which the host cannot see (the sequence lengths are
  // on the device), and slower on short ones
  if (t_kernel == kKernAb) return kKernAb;
  const int64_t cpt = cands_per_tile(Lq);
  const int64_t pair = 2 * cpt;        // candidates of a two-tile item
  const bool two_tiles = n_cand >= pair * n_user;
  const int64_t items = int64_t(H) * ((n_cand + pair - 1) / pair);
  const bool late_clc = target_only && D == 128 && n_user <= kClcMaxUsers;
  return (two_tiles && items >= (late_clc ? kPpMinItemsClc : kPpMinItems)) ? kKernPp : kKernTc;
}

// The kernel a call runs.  self_T >= 0: a fused self + target call, which
// runs on the one- or two-tile kernel.
int effective_kernel(int64_t n_cand, int64_t n_user, int H, int Lq, int D, int64_t self_T) {
  const int k = kernel_choice(n_cand, n_user, H, Lq, D, self_T < 0);
  return (self_T >= 0 && (k == kKernSimt || k == kKernAb)) ? kKernTc : k;
}

// kernel: kKernTc (plans in-kernel when the inputs fit its shared memory,
// otherwise reads the planning kernel's list; never splits a unit through
// global memory), kKernPp (always plans in-kernel), kKernSimt (planning
// kernel, may split).
// extra_units: further work items the in-kernel planning may make (the
// self-attention tiles of a fused call).
// multi_level: a user -> vendor -> item call; when the planning kernel plans
// it, it writes every item's user to item_user first.
Workspace plan_workspace(int64_t n_cand, int64_t n_user, int H, int Lq, int D, int num_sms,
                         int grid, int kernel, int64_t extra_units = 0, bool multi_level = false,
                         bool clc = false) {
  Workspace w = {};
  w.clc = clc;
  const int cpt = cands_per_tile(Lq);
  const int64_t units_bound =
      int64_t(H) * ((n_cand + cpt - 1) / cpt + (n_user < n_cand ? n_user : n_cand)) + extra_units;
  w.grid = grid;
  w.kernel = kernel;
  // keep in step with ikbo_launches_per_call
  w.fused = kernel != kKernSimt && fits_in_kernel_planning(n_cand, n_user);
  w.max_items = int(num_sms + units_bound);
  w.max_split_items = kernel == kKernSimt ? 3 * num_sms : 0;
  w.max_units = w.max_split_items;
  w.max_cta_items = int((units_bound + grid - 1) / grid) + 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  w.header = take(sizeof(PlanHeader));
  w.perm = take(sizeof(int32_t) * size_t(n_cand));
  // per CTA: the K and V maps with the row count T, then one bounded V map per work item
  const int64_t listed_per_cta = (int64_t(w.max_items) + grid - 1) / grid;
  w.map_stride = 2 + int(listed_per_cta > w.max_cta_items ? listed_per_cta : w.max_cta_items);
  w.map_slots = take(sizeof(CUtensorMap) * size_t(grid) * size_t(w.map_stride));
  if (w.fused && w.clc) {
    // per SM: offsets, first candidates, units before each rank, users by
    // rank (n_user + 1 ints each), then one bounded V map per user
    w.clc_map_offset = int(align_up(sizeof(int32_t) * 4 * size_t(n_user + 1), 128));
    w.clc_slot_bytes = int(w.clc_map_offset + sizeof(CUtensorMap) * size_t(n_user));
    w.clc_slots = take(size_t(kClcSlots) * size_t(w.clc_slot_bytes));
  }
  if (w.fused) {
    w.cta_items = take(sizeof(WorkItem) * size_t(grid) * size_t(w.max_cta_items));
    if (kernel == kKernAb) {
      // partial results of units cut into key-range chunks: one chunk per CTA
      w.ab_o = take(sizeof(float) * size_t(grid) * kTileM * D);
      w.ab_lse = take(sizeof(float) * size_t(grid) * kTileM);
      w.ab_flags = take(sizeof(unsigned long long) * size_t(grid));
    }
  } else {
    w.kmap = take(sizeof(CUtensorMap));
    w.vmap = take(sizeof(CUtensorMap));
    w.items = take(sizeof(WorkItem) * size_t(w.max_items));
    w.units = take(sizeof(UnitInfo) * size_t(w.max_units > 0 ? w.max_units : 1));
    w.cand_start = take(sizeof(int32_t) * size_t(n_user + 1));
    w.scratch = take(sizeof(int32_t) * size_t(3 * n_user + 2));
    if (multi_level) w.item_user = take(sizeof(int32_t) * size_t(n_cand));
    if (w.max_split_items) {
      w.partial_o = take(sizeof(float) * size_t(w.max_split_items) * kTileM * D);
      w.partial_ml = take(sizeof(float2) * size_t(w.max_split_items) * kTileM);
    }
  }
  w.total = o;
  return w;
}

// Row count of the K/V maps that the tcgen05 kernel loads through directly
// when it plans in-kernel: open, since T is only known on the device.  Every
// tile it loads this way lies inside rows [0, T); a tile that reaches past T
// goes through a device-side copy with the row count set to T.
constexpr cuuint64_t kOpenRows = 0x7fffffff;

int encode_kv_map(CUtensorMap* m, const void* base, int H, int D, int block_n, cuuint64_t rows) {
  // 2-D view of k (or v): rows = tokens, columns = H * D.  `rows` is either
  // open (above) or a placeholder that the planning kernel replaces with T.
  cuuint64_t dims[2] = {cuuint64_t(H) * D, rows};
  cuuint64_t strides[1] = {cuuint64_t(H) * D * 2};
  cuuint32_t box[2] = {64, cuuint32_t(block_n)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IKBO_OK : IKBO_ERR_CUDA;
}

int encode_q_map(CUtensorMap* m, const void* q, int64_t n_cand, int H, int Lq, int D, int nb) {
  // 4-D view {D, Lq, H, n_cand}; one box = nb candidates x Lq tokens x 64
  // columns of one head, as 128-byte swizzled rows.
  cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Lq), cuuint64_t(H), cuuint64_t(n_cand)};
  cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(Lq) * D * 2, cuuint64_t(H) * Lq * D * 2};
  cuuint32_t box[4] = {64, cuuint32_t(Lq), 1, cuuint32_t(nb)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IKBO_OK : IKBO_ERR_CUDA;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  return launch_ex(kern, grid, block, smem, st, true, 1, args...);
}

// CTAs of the tcgen05 kernel: two per cluster, as many clusters as fit at once.
template <int D>
int tc_grid(DeviceState* ds) {
  int& g = ds->tc_grid[D == 128 ? 1 : 0];
  if (g) return g;
  if (cudaFuncSetAttribute(ikbo_attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(ikbo_attn_tc_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           0) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ds->num_sms & ~1);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, ikbo_attn_tc_kernel<D>, &cfg) != cudaSuccess ||
      clusters <= 0) {
    cudaGetLastError();
    clusters = ds->num_sms / 2;
  }
  g = 2 * clusters;
  return g;
}

// CTAs of the key-interleaved kernel: one per SM, no clusters, all resident
// at once (a unit cut into chunks is merged by a CTA that waits for the others).
template <int D>
int ab_grid(DeviceState* ds) {
  int& g = ds->ab_grid[D == 128 ? 1 : 0];
  if (g) return g;
  if (cudaFuncSetAttribute(ikbo_attn_ab_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmemBytes) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ikbo_attn_ab_kernel<D>, kTcThreads,
                                                    kTcSmemBytes) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    return 0;
  }
  g = ds->num_sms * per_sm;
  return g;
}

// CTAs of the two-tile kernel: one per SM, no clusters.
template <int D>
int pp_grid(DeviceState* ds) {
  int& g = ds->pp_grid[D == 128 ? 1 : 0];
  if (g) return g;
  if (cudaFuncSetAttribute(ikbo_attn_pp_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(ikbo_attn_pp_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTcSmemBytes) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ikbo_attn_pp_kernel<D, false>, kTcThreads,
                                                    kTcSmemBytes) != cudaSuccess ||
      per_sm <= 0) {
    cudaGetLastError();
    per_sm = 1;
  }
  g = ds->num_sms * per_sm;
  return g;
}

template <int D>
cudaError_t launch_attn_tc(const AttnParams& ap, const CUtensorMap& qmap, const CUtensorMap& qmap1,
                           const CUtensorMap& kt, const CUtensorMap& vt, const CUtensorMap& qut,
                           int grid, bool pdl, cudaStream_t st) {
  return launch_ex(ikbo_attn_tc_kernel<D>, dim3(grid), dim3(kTcThreads), kTcSmemBytes, st, pdl, 2,
                   ap, qmap, qmap1, kt, vt, qut);
}

template <int D>
cudaError_t launch_attn_ab(const AttnParams& ap, const CUtensorMap& qmap, const CUtensorMap& qmap1,
                           const CUtensorMap& kt, const CUtensorMap& vt, int grid, cudaStream_t st) {
  return launch_ex(ikbo_attn_ab_kernel<D>, dim3(grid), dim3(kTcThreads), kTcSmemBytes, st, false, 1, ap,
                   qmap, qmap1, kt, vt);
}

template <int D>
cudaError_t launch_attn_pp(const AttnParams& ap, const CUtensorMap& qmap, const CUtensorMap& qmap1,
                           const CUtensorMap& kt, const CUtensorMap& vt, const CUtensorMap& qut,
                           int grid, cudaStream_t st) {
  // the fused self + target form only for fused calls
  if (ap.q_user)
    return launch_ex(ikbo_attn_pp_kernel<D, true>, dim3(grid), dim3(kTcThreads), kTcSmemBytes, st, false,
                     1, ap, qmap, qmap1, kt, vt, qut);
  return launch_ex(ikbo_attn_pp_kernel<D, false>, dim3(grid), dim3(kTcThreads), kTcSmemBytes, st, false, 1,
                   ap, qmap, qmap1, kt, vt, qut);
}

// The self-attention part of a fused call: the user sequence's queries and
// output, [T, H, D] each.
struct SelfPart {
  const void* q_user;
  void* out_user;
  int64_t T;
};

// The vendor level of a multi-level call: c2u then holds item_to_vendor.
struct VendorLevel {
  const int32_t* vendor_to_user;
  int64_t n_vendor;
};

// Plan + attention on device buffers, scratch from `ws` (>= plan_workspace().total).
int run_ikbo(DeviceState* ds, const void* q, const void* k, const void* v, const int32_t* off,
             const int32_t* c2u, int64_t n_cand, int64_t n_user, int H, int Lq, int D, float scale,
             void* out, char* ws, const Workspace& L, cudaStream_t st,
             const SelfPart* self = nullptr, const VendorLevel* vendor = nullptr) {
  const int kernel = L.kernel;
  PlanParams pp = {};
  pp.cand_to_user = c2u;
  pp.user_offsets = off;
  pp.n_cand = n_cand;
  pp.n_user = n_user;
  pp.H = H;
  pp.cands_per_tile = cands_per_tile(Lq);
  pp.block_n = kBlockN;
  pp.num_sms = ds->num_sms;
  pp.max_items = L.max_items;
  pp.max_split_items = L.max_split_items;
  pp.max_units = L.max_units;
  pp.allow_split = kernel == kKernSimt ? 1 : 0;
  pp.header = reinterpret_cast<PlanHeader*>(ws + L.header);
  pp.items = reinterpret_cast<WorkItem*>(ws + L.items);
  pp.units = reinterpret_cast<UnitInfo*>(ws + L.units);
  pp.perm = reinterpret_cast<int32_t*>(ws + L.perm);
  pp.cand_start = reinterpret_cast<int32_t*>(ws + L.cand_start);
  pp.scratch = reinterpret_cast<int32_t*>(ws + L.scratch);
  pp.err_word = error_word(ds, st);
  if (vendor) {
    pp.vendor_to_user = vendor->vendor_to_user;
    pp.n_vendor = vendor->n_vendor;
    pp.item_user = reinterpret_cast<int32_t*>(ws + L.item_user);
  }

  PlanExtra px;
  std::memset(&px, 0, sizeof px);
  px.out = out;
  px.Lq = Lq;
  px.D = D;
  px.patch_maps = kernel != kKernSimt ? 1 : 0;
  px.kmap_dst = reinterpret_cast<CUtensorMap*>(ws + L.kmap);
  px.vmap_dst = reinterpret_cast<CUtensorMap*>(ws + L.vmap);
  CUtensorMap qmap, qmap1, qumap;
  std::memset(&qmap, 0, sizeof qmap);
  std::memset(&qmap1, 0, sizeof qmap1);
  std::memset(&qumap, 0, sizeof qumap);
  if (kernel != kKernSimt) {
    // A fused call states T: its maps carry the row count itself.  Otherwise
    // in-kernel planning loads through open maps (T is only known on the
    // device), and the planning kernel patches a placeholder.
    const cuuint64_t rows = self ? cuuint64_t(self->T > 0 ? self->T : 1)
                                 : (L.fused ? kOpenRows : cuuint64_t(kBlockN));
    if (encode_kv_map(&px.kmap_tmpl, k, H, D, kBlockN, rows) != IKBO_OK ||
        encode_kv_map(&px.vmap_tmpl, v, H, D, kBlockN, rows) != IKBO_OK)
      return IKBO_ERR_CUDA;
    if (n_cand > 0 && (encode_q_map(&qmap, q, n_cand, H, Lq, D, qbox_cands(Lq)) != IKBO_OK ||
                       encode_q_map(&qmap1, q, n_cand, H, Lq, D, 1) != IKBO_OK))
      return IKBO_ERR_CUDA;
    if (self && self->T > 0 && encode_kv_map(&qumap, self->q_user, H, D, kBlockN, rows) != IKBO_OK)
      return IKBO_ERR_CUDA;
  }

  AttnParams ap = {};
  ap.q = static_cast<const uint16_t*>(q);
  ap.k = static_cast<const uint16_t*>(k);
  ap.v = static_cast<const uint16_t*>(v);
  ap.out = static_cast<uint16_t*>(out);
  ap.n_cand = n_cand;
  ap.H = H;
  ap.Lq = Lq;
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.max_items = L.max_items;
  ap.header = pp.header;
  ap.items = pp.items;
  ap.units = pp.units;
  ap.perm = pp.perm;
  ap.partial_o = L.max_split_items ? reinterpret_cast<float*>(ws + L.partial_o) : nullptr;
  ap.partial_ml = L.max_split_items ? reinterpret_cast<float2*>(ws + L.partial_ml) : nullptr;
  ap.err_word = error_word(ds, st);
  ap.kmap = px.kmap_dst;
  ap.vmap = px.vmap_dst;
  ap.timeout_ns = g_timeout_ns;
  ap.qbox = qbox_cands(Lq);
  ap.debug_flags = g_debug_flags;
  ap.trace = g_trace;
  ap.trace_ctas = ds->num_sms;
  ap.fused = L.fused ? 1 : 0;
  ap.cands_per_tile = pp.cands_per_tile;
  ap.user_offsets = off;
  ap.cand_to_user = c2u;
  ap.n_user = n_user;
  ap.cta_items = reinterpret_cast<WorkItem*>(ws + L.cta_items);
  ap.max_cta_items = L.max_cta_items;
  ap.perm_ws = pp.perm;
  ap.map_slots = reinterpret_cast<CUtensorMap*>(ws + L.map_slots);
  ap.map_stride = L.map_stride;
  if (L.clc) {
    ap.clc = 1;
    // the prologue stamps (flag 4) of every CTA are not bounded by the trace
    // buffer's CTAs, and this grid has more CTAs than SMs
    ap.debug_flags &= ~4;
    ap.clc_slots = reinterpret_cast<uint8_t*>(ws + L.clc_slots);
    ap.clc_slot_bytes = L.clc_slot_bytes;
    ap.clc_map_offset = L.clc_map_offset;
  }
  if (kernel == kKernAb) {
    ap.ab_partial_o = reinterpret_cast<float4*>(ws + L.ab_o);
    ap.ab_partial_lse = reinterpret_cast<float*>(ws + L.ab_lse);
    ap.ab_flags = reinterpret_cast<unsigned long long*>(ws + L.ab_flags);
    ap.ab_marker = ((ds->calls->fetch_add(1) + 1) << 1) | 1ull;
  }
  if (self) {
    ap.q_user = static_cast<const uint16_t*>(self->q_user);
    ap.out_user = static_cast<uint16_t*>(self->out_user);
    ap.total_rows = self->T;
    ap.exact_rows = 1;
  }
  if (vendor) {
    ap.vendor_to_user = vendor->vendor_to_user;
    ap.n_vendor = vendor->n_vendor;
  }

  const bool timed = g_timing;
  if (timed) cudaEventRecord(ds->ev[0], st);
  if (!L.fused) {
    ikbo_plan_kernel<<<1, kPlanThreads, 0, st>>>(pp, px);
    if (cudaGetLastError() != cudaSuccess) return IKBO_ERR_CUDA;
  }
  if (timed) cudaEventRecord(ds->ev[1], st);
  cudaError_t e;
  if (kernel == kKernSimt) {
    const int grid = L.max_items < ds->num_sms * 8 ? L.max_items : ds->num_sms * 8;
    if (D == 64)
      e = launch_pdl(ikbo_attn_simt_kernel<64>, dim3(grid), dim3(kSimtThreads), 0, st, ap);
    else
      e = launch_pdl(ikbo_attn_simt_kernel<128>, dim3(grid), dim3(kSimtThreads), 0, st, ap);
  } else if (kernel == kKernAb) {
    if (D == 64)
      e = launch_attn_ab<64>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, L.grid, st);
    else
      e = launch_attn_ab<128>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, L.grid, st);
  } else if (kernel == kKernPp) {
    if (D == 64)
      e = launch_attn_pp<64>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, qumap, L.grid, st);
    else
      e = launch_attn_pp<128>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, qumap, L.grid, st);
  } else {
    // the planning kernel (listed mode) is followed with programmatic dependent launch
    if (D == 64)
      e = launch_attn_tc<64>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, qumap, L.grid, !L.fused, st);
    else
      e = launch_attn_tc<128>(ap, qmap, qmap1, px.kmap_tmpl, px.vmap_tmpl, qumap, L.grid, !L.fused, st);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (timed) {
    cudaEventRecord(ds->ev[2], st);
    int dev = 0;
    cudaGetDevice(&dev);
    g_timing_dev = dev;
  }
  return IKBO_OK;
}

// Workspace for a call on this device with the current kernel choice.
// self_T >= 0: a fused self + target call over T sequence rows, which a
// tcgen05 kernel runs with its planning in-kernel (the one-tile kernel when
// the choice is the SIMT kernel).
int call_workspace(DeviceState* ds, int64_t n_cand, int64_t n_user, int H, int Lq, int D,
                   Workspace* out, int64_t self_T = -1, bool multi_level = false) {
  int grid = 0;
  const int kernel = effective_kernel(n_cand, n_user, H, Lq, D, self_T);
  if (kernel == kKernAb) {
    grid = D == 64 ? ab_grid<64>(ds) : ab_grid<128>(ds);
    if (grid <= 0) return IKBO_ERR_CUDA;
  } else if (kernel == kKernTc) {
    grid = D == 64 ? tc_grid<64>(ds) : tc_grid<128>(ds);
    if (grid <= 0) return IKBO_ERR_CUDA;
  } else if (kernel == kKernPp) {
    grid = D == 64 ? pp_grid<64>(ds) : pp_grid<128>(ds);
    if (grid <= 0) return IKBO_ERR_CUDA;
  }
  // a self-attention tile per 128 rows of every user, at most T / 128 + n_user per head
  const int64_t extra = self_T > 0 ? int64_t(H) * ((self_T + kTileM - 1) / kTileM + n_user) : 0;
  const bool clc = kernel == kKernPp && self_T < 0 && n_user <= kClcMaxUsers;
  if (clc) {
    const int64_t ub = pp_units_bound(n_cand, n_user, H, Lq);
    grid = int(ub > 0 ? ub : 1);
  }
  *out = plan_workspace(n_cand, n_user, H, Lq, D, ds->num_sms, grid > 0 ? grid : ds->num_sms,
                        kernel, extra, multi_level, clc);
  return IKBO_OK;
}

int ensure_events(DeviceState* ds) {
  if (ds->ev_ready) return IKBO_OK;
  for (auto& e : ds->ev)
    if (cudaEventCreate(&e) != cudaSuccess) return IKBO_ERR_CUDA;
  ds->ev_ready = true;
  return IKBO_OK;
}

}  // namespace
}  // namespace ikbo

using namespace ikbo;

extern "C" {

int ikbo_attn_fwd(const void* q, const void* k_user, const void* v_user,
                  const int32_t* user_offsets, const int32_t* cand_to_user, int64_t n_cand,
                  int64_t n_user, int32_t H, int32_t Lq, int32_t D, float scale, void* out,
                  ikbo_stream_t stream) {
  int rc = check_args(q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK || n_cand == 0) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Workspace L;
  if ((rc = call_workspace(ds, n_cand, n_user, H, Lq, D, &L)) != IKBO_OK) return rc;
  void* ws = nullptr;
  if (pool_alloc(ds, &ws, L.total, st) != cudaSuccess) return IKBO_ERR_CUDA;
  rc = run_ikbo(ds, q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D, scale,
                out, static_cast<char*>(ws), L, st);
  if (cudaFreeAsync(ws, st) != cudaSuccess && rc == IKBO_OK) rc = IKBO_ERR_CUDA;
  return rc;
}

// Status of a device error word (0 = none).
int status_of_error_word(int word) {
  if (word & kErrIndex) return IKBO_ERR_INDEX;
  if (word & kErrOffsets) return IKBO_ERR_OFFSETS;
  if (word & kErrTimeout) return IKBO_ERR_TIMEOUT;
  if (word & kErrLayout) return IKBO_ERR_CUDA;
  return IKBO_OK;
}

int ikbo_attn_fwd_host(const void* q, const void* k_user, const void* v_user,
                       const int32_t* user_offsets, const int32_t* cand_to_user, int64_t n_cand,
                       int64_t n_user, int32_t H, int32_t Lq, int32_t D, float scale, void* out,
                       ikbo_stream_t stream) {
  int rc = check_args(q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK || n_cand == 0) return rc;
  if (user_offsets[0] != 0) return IKBO_ERR_OFFSETS;
  const int64_t T = user_offsets[n_user];
  if (T < 0) return IKBO_ERR_OFFSETS;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Workspace L;
  if ((rc = call_workspace(ds, n_cand, n_user, H, Lq, D, &L)) != IKBO_OK) return rc;
  const size_t qbytes = size_t(n_cand) * H * Lq * D * 2;
  const size_t kvbytes = size_t(T) * H * D * 2;
  const size_t o_q = 0, o_k = align_up(o_q + qbytes, 256), o_v = align_up(o_k + kvbytes, 256);
  const size_t o_off = align_up(o_v + kvbytes, 256);
  const size_t o_c2u = align_up(o_off + size_t(n_user + 1) * 4, 256);
  const size_t o_out = align_up(o_c2u + size_t(n_cand) * 4, 256);
  const size_t o_ws = align_up(o_out + qbytes, 256);
  char* buf = nullptr;
  if (pool_alloc(ds, &buf, o_ws + L.total, st) != cudaSuccess)
    return IKBO_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMemcpyAsync(buf + o_q, q, qbytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && kvbytes) e = cudaMemcpyAsync(buf + o_k, k_user, kvbytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && kvbytes) e = cudaMemcpyAsync(buf + o_v, v_user, kvbytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(buf + o_off, user_offsets, size_t(n_user + 1) * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(buf + o_c2u, cand_to_user, size_t(n_cand) * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) {
    rc = run_ikbo(ds, buf + o_q, buf + o_k, buf + o_v, reinterpret_cast<int32_t*>(buf + o_off),
                  reinterpret_cast<int32_t*>(buf + o_c2u), n_cand, n_user, H, Lq, D, scale,
                  buf + o_out, buf + o_ws, L, st);
    if (rc == IKBO_OK) e = cudaMemcpyAsync(out, buf + o_out, qbytes, cudaMemcpyDeviceToHost, st);
  }
  cudaFreeAsync(buf, st);
  // the device error word comes back with the output, under the same
  // synchronisation (a pinned word per device, made on the first such call;
  // one host call at a time)
  std::lock_guard<std::mutex> lock(*ds->host_call);
  if (!ds->err_host) {
    void* h = nullptr;
    if (cudaHostAlloc(&h, sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
      cudaStreamSynchronize(st);
      return IKBO_ERR_CUDA;
    }
    ds->err_host = static_cast<int*>(h);
  }
  int* const word_dev = error_word(ds, st);
  if (e == cudaSuccess && rc == IKBO_OK)
    e = cudaMemcpyAsync(ds->err_host, word_dev, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (cudaStreamSynchronize(st) != cudaSuccess || e != cudaSuccess) return IKBO_ERR_CUDA;
  if (rc != IKBO_OK) return rc;
  const int word = *ds->err_host;
  if (word) {
    // clear it, as ikbo_get_device_error does
    if (cudaMemsetAsync(word_dev, 0, sizeof(int), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return IKBO_ERR_CUDA;
  }
  return status_of_error_word(word);
}

int ikbo_broadcast_attn_fwd(const void* q, const void* k_user, const void* v_user,
                            const int32_t* user_offsets, const int32_t* cand_to_user,
                            int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                            float scale, void* out, size_t mem_budget_bytes,
                            ikbo_stream_t stream) {
  int rc = check_args(q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK || n_cand == 0) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Read the index tensors back to size the copies.
  std::vector<int32_t> off(static_cast<size_t>(n_user + 1));
  std::vector<int32_t> c2u(static_cast<size_t>(n_cand));
  if (cudaMemcpyAsync(off.data(), user_offsets, off.size() * 4, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(c2u.data(), cand_to_user, c2u.size() * 4, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return IKBO_ERR_CUDA;
  if (off[0] != 0) return IKBO_ERR_OFFSETS;
  for (int64_t u = 0; u < n_user; ++u)
    if (off[u + 1] < off[u]) return IKBO_ERR_OFFSETS;
  for (int64_t c = 0; c < n_cand; ++c)
    if (c2u[c] < 0 || c2u[c] >= n_user) return IKBO_ERR_INDEX;
  const size_t row_bytes = size_t(H) * D * 2;
  const size_t qrow = size_t(H) * Lq * D * 2;
  // Chunks [c0, c1) whose K+V copy fits the budget.
  std::vector<int64_t> cuts(1, 0);
  std::vector<int64_t> chunk_rows;
  {
    int64_t rows = 0;
    for (int64_t c = 0; c < n_cand; ++c) {
      const int64_t L = off[c2u[c] + 1] - off[c2u[c]];
      if (size_t(L) * row_bytes * 2 > mem_budget_bytes) return IKBO_ERR_BUDGET;
      if (size_t(rows + L) * row_bytes * 2 > mem_budget_bytes) {
        cuts.push_back(c);
        chunk_rows.push_back(rows);
        rows = 0;
      }
      rows += L;
    }
    cuts.push_back(n_cand);
    chunk_rows.push_back(rows);
  }
  // Per candidate: source row, destination offset (int64, copy kernel) and
  // the per-chunk jagged offsets / identity map (int32, attention), all
  // copied to the device once.
  std::vector<int32_t> src(static_cast<size_t>(n_cand));
  std::vector<int32_t> offb(static_cast<size_t>(n_cand) + cuts.size());
  std::vector<int32_t> id(static_cast<size_t>(n_cand));
  std::vector<int64_t> dst(static_cast<size_t>(n_cand) + cuts.size());
  {
    size_t ob = 0;
    for (size_t ch = 0; ch + 1 < cuts.size(); ++ch) {
      int64_t acc = 0;
      for (int64_t c = cuts[ch]; c < cuts[ch + 1]; ++c) {
        const int32_t u = c2u[c];
        src[c] = off[u];
        dst[ob] = acc;
        offb[ob] = int32_t(acc);
        id[c] = int32_t(c - cuts[ch]);
        acc += off[u + 1] - off[u];
        ++ob;
      }
      dst[ob] = acc;
      offb[ob] = int32_t(acc);
      ++ob;
    }
  }
  const size_t m_src = 0, m_dst = align_up(src.size() * 4, 256);
  const size_t m_offb = align_up(m_dst + dst.size() * 8, 256);
  const size_t m_id = align_up(m_offb + offb.size() * 4, 256);
  const size_t m_total = align_up(m_id + id.size() * 4, 256);
  char* meta = nullptr;
  if (pool_alloc(ds, &meta, m_total, st) != cudaSuccess)
    return IKBO_ERR_CUDA;
  cudaError_t e = cudaMemcpyAsync(meta + m_src, src.data(), src.size() * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(meta + m_dst, dst.data(), dst.size() * 8, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(meta + m_offb, offb.data(), offb.size() * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(meta + m_id, id.data(), id.size() * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // host vectors die at return
  if (e != cudaSuccess) {
    cudaFreeAsync(meta, st);
    return IKBO_ERR_CUDA;
  }
  const bool timed = g_timing;
  if (timed) {
    if ((rc = ensure_events(ds)) != IKBO_OK) {
      cudaFreeAsync(meta, st);
      return rc;
    }
    cudaEventRecord(ds->ev[0], st);
    cudaEventRecord(ds->ev[1], st);
  }
  g_timing = false;   // the inner attention calls must not move the events
  size_t ob = 0;
  for (size_t ch = 0; ch + 1 < cuts.size() && rc == IKBO_OK; ++ch) {
    const int64_t c0 = cuts[ch], n = cuts[ch + 1] - c0, rows = chunk_rows[ch];
    Workspace L;
    if ((rc = call_workspace(ds, n, n, H, Lq, D, &L)) != IKBO_OK) break;
    const size_t o_kb = 0, o_vb = align_up(size_t(rows) * row_bytes, 256);
    const size_t o_ws = align_up(o_vb + size_t(rows) * row_bytes, 256);
    char* buf = nullptr;
    if (pool_alloc(ds, &buf, o_ws + L.total, st) != cudaSuccess) {
      rc = IKBO_ERR_CUDA;
      break;
    }
    const int grid = int(n < 4 * ds->num_sms ? n : 4 * ds->num_sms);
    ikbo_broadcast_copy_kernel<<<grid, 256, 0, st>>>(
        static_cast<const uint4*>(k_user), static_cast<const uint4*>(v_user),
        reinterpret_cast<uint4*>(buf + o_kb), reinterpret_cast<uint4*>(buf + o_vb),
        reinterpret_cast<const int32_t*>(meta + m_src) + c0,
        reinterpret_cast<const int64_t*>(meta + m_dst) + ob, int32_t(n), int32_t(row_bytes / 16));
    if (cudaGetLastError() != cudaSuccess) rc = IKBO_ERR_CUDA;
    if (rc == IKBO_OK)
      rc = run_ikbo(ds, static_cast<const char*>(q) + size_t(c0) * qrow, buf + o_kb, buf + o_vb,
                    reinterpret_cast<int32_t*>(meta + m_offb) + ob,
                    reinterpret_cast<int32_t*>(meta + m_id) + c0, n, n, H, Lq, D, scale,
                    static_cast<char*>(out) + size_t(c0) * qrow, buf + o_ws, L, st);
    cudaFreeAsync(buf, st);
    ob += size_t(n) + 1;
  }
  g_timing = timed;
  if (timed) {
    cudaEventRecord(ds->ev[2], st);
    int dev = 0;
    cudaGetDevice(&dev);
    g_timing_dev = dev;
  }
  cudaFreeAsync(meta, st);
  return rc;
}

int ikbo_fused_attn_fwd(const void* q, const void* q_user, const void* k_user, const void* v_user,
                        const int32_t* user_offsets, const int32_t* cand_to_user, int64_t n_cand,
                        int64_t n_user, int64_t T, int32_t H, int32_t Lq, int32_t D, float scale,
                        void* out, void* out_user, ikbo_stream_t stream) {
  if (T < 0 || T >= (int64_t(1) << 31)) return IKBO_ERR_SHAPE;
  int rc = check_args(q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK) return rc;
  if (n_cand == 0 && T == 0) return IKBO_OK;
  if (T > 0) {
    if (!q_user || !out_user || !k_user || !v_user || !user_offsets) return IKBO_ERR_NULL;
    if (!aligned16(q_user) || !aligned16(out_user) || !aligned16(k_user) || !aligned16(v_user) ||
        (reinterpret_cast<uintptr_t>(user_offsets) & 3u))
      return IKBO_ERR_ALIGN;
    // out_user may share no byte with an input or with out
    const uintptr_t ub = reinterpret_cast<uintptr_t>(out_user);
    const uintptr_t ue = ub + uintptr_t(T) * H * D * 2;
    auto overlaps = [&](const void* x, uintptr_t bytes) {
      const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
      return x && xb < ue && ub < xb + bytes;
    };
    const uintptr_t seq = uintptr_t(T) * H * D * 2, cand = uintptr_t(n_cand) * H * Lq * D * 2;
    if (overlaps(q_user, seq) || overlaps(k_user, seq) || overlaps(v_user, seq) ||
        (n_cand > 0 && (overlaps(q, cand) || overlaps(out, cand))))
      return IKBO_ERR_ALIAS;
  }
  if (!fits_in_kernel_planning(n_cand, n_user)) return IKBO_ERR_SHAPE;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Workspace L;
  if ((rc = call_workspace(ds, n_cand, n_user, H, Lq, D, &L, T)) != IKBO_OK) return rc;
  void* ws = nullptr;
  if (pool_alloc(ds, &ws, L.total, st) != cudaSuccess) return IKBO_ERR_CUDA;
  const SelfPart self{q_user, out_user, T};
  rc = run_ikbo(ds, q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D, scale,
                out, static_cast<char*>(ws), L, st, &self);
  if (cudaFreeAsync(ws, st) != cudaSuccess && rc == IKBO_OK) rc = IKBO_ERR_CUDA;
  return rc;
}

int ikbo_ml_attn_fwd(const void* q, const void* k_user, const void* v_user,
                     const int32_t* user_offsets, const int32_t* item_to_vendor,
                     const int32_t* vendor_to_user, int64_t n_item, int64_t n_vendor,
                     int64_t n_user, int32_t H, int32_t Lq, int32_t D, float scale, void* out,
                     ikbo_stream_t stream) {
  if (n_vendor < 0 || n_vendor >= (int64_t(1) << 31)) return IKBO_ERR_SHAPE;
  int rc = check_args(q, k_user, v_user, user_offsets, item_to_vendor, n_item, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK || n_item == 0) return rc;
  if (!vendor_to_user) return IKBO_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(vendor_to_user) & 3u) return IKBO_ERR_ALIGN;
  if (n_vendor == 0) return IKBO_ERR_INDEX;   // every item would name a vendor outside [0, 0)
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Workspace L;
  if ((rc = call_workspace(ds, n_item, n_user, H, Lq, D, &L, -1, true)) != IKBO_OK) return rc;
  void* ws = nullptr;
  if (pool_alloc(ds, &ws, L.total, st) != cudaSuccess) return IKBO_ERR_CUDA;
  const VendorLevel vendor{vendor_to_user, n_vendor};
  rc = run_ikbo(ds, q, k_user, v_user, user_offsets, item_to_vendor, n_item, n_user, H, Lq, D,
                scale, out, static_cast<char*>(ws), L, st, nullptr, &vendor);
  if (cudaFreeAsync(ws, st) != cudaSuccess && rc == IKBO_OK) rc = IKBO_ERR_CUDA;
  return rc;
}

}  // extern "C"

namespace ikbo {
namespace {

// W [M, K] row-major as a 2-D map {K, M}: boxes of 64 K-columns x 128 rows.
int encode_lce_w_map(CUtensorMap* m, const void* W, int M, int K) {
  cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(M)};
  cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  cuuint32_t box[2] = {cuuint32_t(kLceKStep), cuuint32_t(kTileM)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IKBO_OK : IKBO_ERR_CUDA;
}

// X [B, K, N] as a 3-D map {N, K, B}: boxes of 64 columns x 64 K-rows of one batch entry.
int encode_lce_x_map(CUtensorMap* m, const void* X, int64_t B, int K, int N) {
  cuuint64_t dims[3] = {cuuint64_t(N), cuuint64_t(K), cuuint64_t(B)};
  cuuint64_t strides[2] = {cuuint64_t(N) * 2, cuuint64_t(K) * N * 2};
  cuuint32_t box[3] = {64, cuuint32_t(kLceKStep), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(X), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IKBO_OK : IKBO_ERR_CUDA;
}

// out [B, M, N] (the output, or the term of the level below) as a 3-D map
// {N, M, B}: the epilogue's store boxes of 64 columns x 32 rows of one entry
// (rows past M are not written).
int encode_lce_out_map(CUtensorMap* m, const void* out, int64_t B, int M, int N) {
  cuuint64_t dims[3] = {cuuint64_t(N), cuuint64_t(M), cuuint64_t(B)};
  cuuint64_t strides[2] = {cuuint64_t(N) * 2, cuuint64_t(M) * N * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(out), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? IKBO_OK : IKBO_ERR_CUDA;
}

// Units of the batch: one per batch entry and row tile, or, with clusters, one
// per batch entry (a cluster of cluster_n CTAs takes its row tiles).  Grid:
// as many CTAs as there are units, at most as many as fit at once.
template <int NB, bool kPair>
cudaError_t launch_lce(DeviceState* ds, const LceParams& lp, const CUtensorMap& wm,
                       const CUtensorMap& xm, bool pdl, cudaStream_t st) {
  CUtensorMap om;
  if (encode_lce_out_map(&om, lp.out, lp.n_batch, lp.M, lp.N) != IKBO_OK) return cudaErrorInvalidValue;
  auto kern = ikbo_lce_kernel<NB, kPair>;
  if (!ds->lce_ready[kPair][NB - 1]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLceSmemBytes);
    if (e != cudaSuccess) return e;
    ds->lce_ready[kPair][NB - 1] = true;
  }
  const int cn = lp.cluster_n;
  int grid = 0;
  if (cn > 1) {
    int& fit = ds->lce_clusters[kPair][NB - 1][cn];
    if (!fit) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((ds->num_sms / cn) * cn);
      cfg.blockDim = dim3(kLceThreads);
      cfg.dynamicSmemBytes = kLceSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cn;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess || fit <= 0) {
        cudaGetLastError();
        fit = ds->num_sms / cn;
      }
    }
    const int64_t clusters = lp.n_batch < fit ? lp.n_batch : fit;
    grid = int(clusters) * cn;
  } else {
    const int64_t units = lp.n_batch * ((lp.M + kTileM - 1) / kTileM);
    grid = int(units < ds->num_sms ? units : ds->num_sms);
  }
  return launch_ex(kern, dim3(grid), dim3(kLceThreads), kLceSmemBytes, st, pdl, cn, lp, wm, xm, om);
}

// CTA pairs (M = 256 MMAs over two CTAs) when M spans two row tiles or more,
// at most eight, and N is a whole number of 128-column halves
bool lce_pairs(int M, int NB) {
  const int mt = (M + kTileM - 1) / kTileM;
  return NB % 2 == 0 && mt >= 2 && mt <= 8;
}

// CTAs per cluster: the row tiles of one batch entry (rounded up to whole
// pairs with CTA pairs), or 1
int lce_cluster_n(int M, int NB) {
  const int mt = (M + kTileM - 1) / kTileM;
  if (lce_pairs(M, NB)) return 2 * ((mt + 1) / 2);
  return (mt > 1 && mt <= 8) ? mt : 1;
}

cudaError_t launch_lce_nb(DeviceState* ds, int NB, const LceParams& lp, const CUtensorMap& wm,
                          const CUtensorMap& xm, bool pdl, cudaStream_t st) {
  if (lce_pairs(lp.M, NB)) {
    if (NB == 2) return launch_lce<2, true>(ds, lp, wm, xm, pdl, st);
    return launch_lce<4, true>(ds, lp, wm, xm, pdl, st);
  }
  switch (NB) {
    case 1: return launch_lce<1, false>(ds, lp, wm, xm, pdl, st);
    case 2: return launch_lce<2, false>(ds, lp, wm, xm, pdl, st);
    case 3: return launch_lce<3, false>(ds, lp, wm, xm, pdl, st);
    default: return launch_lce<4, false>(ds, lp, wm, xm, pdl, st);
  }
}

}  // namespace
}  // namespace ikbo

extern "C" {

int ikbo_lce_fwd(const void* W_user, const void* W_cand, const void* X_user, const void* X_cand,
                 const int32_t* cand_to_user, int64_t n_cand, int64_t n_user, int32_t M,
                 int32_t K_user, int32_t K_cand, int32_t N, void* out, ikbo_stream_t stream) {
  if (n_cand < 0 || n_user < 0 || M < 1 || K_user < 0 || K_cand < 8 || (K_user % 8) ||
      (K_cand % 8) || N < 64 || N > 256 || (N % 64))
    return IKBO_ERR_SHAPE;
  if (n_cand >= (int64_t(1) << 31) || n_user >= (int64_t(1) << 31) || M >= (1 << 24) ||
      K_user >= (1 << 24) || K_cand >= (1 << 24))
    return IKBO_ERR_SHAPE;
  if (n_cand == 0) return IKBO_OK;
  const bool user_part = K_user > 0;
  if (!W_cand || !X_cand || !out || (user_part && (!W_user || !X_user || !cand_to_user)))
    return IKBO_ERR_NULL;
  if (user_part && n_user == 0) return IKBO_ERR_INDEX;
  if (!aligned16(W_cand) || !aligned16(X_cand) || !aligned16(out) ||
      (user_part && (!aligned16(W_user) || !aligned16(X_user) ||
                     (reinterpret_cast<uintptr_t>(cand_to_user) & 3u))))
    return IKBO_ERR_ALIGN;
  {
    const uintptr_t ob = reinterpret_cast<uintptr_t>(out), oe = ob + uintptr_t(n_cand) * M * N * 2;
    auto overlaps = [&](const void* x, uintptr_t bytes) {
      const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
      return x && xb < oe && ob < xb + bytes;
    };
    if (overlaps(W_cand, uintptr_t(M) * K_cand * 2) || overlaps(X_cand, uintptr_t(n_cand) * K_cand * N * 2) ||
        (user_part && (overlaps(W_user, uintptr_t(M) * K_user * 2) ||
                       overlaps(X_user, uintptr_t(n_user) * K_user * N * 2))))
      return IKBO_ERR_ALIAS;
  }
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int NB = N / 64;
  CUtensorMap wc_map, xc_map, wu_map, xu_map;
  std::memset(&wu_map, 0, sizeof wu_map);
  std::memset(&xu_map, 0, sizeof xu_map);
  if (encode_lce_w_map(&wc_map, W_cand, M, K_cand) != IKBO_OK ||
      encode_lce_x_map(&xc_map, X_cand, n_cand, K_cand, N) != IKBO_OK)
    return IKBO_ERR_CUDA;
  uint16_t* Y = nullptr;
  if (user_part) {
    if (encode_lce_w_map(&wu_map, W_user, M, K_user) != IKBO_OK ||
        encode_lce_x_map(&xu_map, X_user, n_user, K_user, N) != IKBO_OK)
      return IKBO_ERR_CUDA;
    if (pool_alloc(ds, &Y, size_t(n_user) * M * N * 2, st) != cudaSuccess)
      return IKBO_ERR_CUDA;
  }
  LceParams lp = {};
  lp.M = M;
  lp.N = N;
  lp.err_word = error_word(ds, st);
  lp.timeout_ns = g_timeout_ns;
  // the row tiles of one batch entry run as one cluster (CTA pairs when N allows)
  lp.cluster_n = lce_cluster_n(M, NB);
  cudaError_t e = cudaSuccess;
  const bool timed = g_timing;
  if (timed && (rc = ensure_events(ds)) != IKBO_OK) {
    if (Y) cudaFreeAsync(Y, st);
    return rc;
  }
  if (timed) cudaEventRecord(ds->ev[0], st);
  if (user_part) {
    LceParams l0 = lp;
    l0.W = static_cast<const uint16_t*>(W_user);
    l0.n_batch = n_user;
    l0.K = K_user;
    l0.out = Y;
    l0.has_dependent = 1;
    e = launch_lce_nb(ds, NB, l0, wu_map, xu_map, false, st);
  }
  if (timed) cudaEventRecord(ds->ev[1], st);
  if (e == cudaSuccess) {
    LceParams l1 = lp;
    l1.W = static_cast<const uint16_t*>(W_cand);
    l1.n_batch = n_cand;
    l1.K = K_cand;
    l1.out = static_cast<uint16_t*>(out);
    l1.add = user_part ? 1 : 0;
    l1.map = cand_to_user;
    l1.n_map = n_user;
    l1.Y = Y;
    // a programmatic dependent of the user stage: its epilogue waits for Y
    e = launch_lce_nb(ds, NB, l1, wc_map, xc_map, user_part, st);
  }
  if (timed) {
    cudaEventRecord(ds->ev[2], st);
    int dev = 0;
    cudaGetDevice(&dev);
    g_timing_dev = dev;
  }
  if (Y) cudaFreeAsync(Y, st);
  return e == cudaSuccess ? IKBO_OK : cuda_fail(e);
}

int ikbo_ml_lce_fwd(const void* W_user, const void* W_vendor, const void* W_item,
                    const void* X_user, const void* X_vendor, const void* X_item,
                    const int32_t* item_to_vendor, const int32_t* vendor_to_user, int64_t n_item,
                    int64_t n_vendor, int64_t n_user, int32_t M, int32_t K_user, int32_t K_vendor,
                    int32_t K_item, int32_t N, void* out, ikbo_stream_t stream) {
  if (n_item < 0 || n_vendor < 0 || n_user < 0 || M < 1 || K_user < 0 || K_vendor < 0 ||
      K_item < 8 || (K_user % 8) || (K_vendor % 8) || (K_item % 8) || N < 64 || N > 256 || (N % 64))
    return IKBO_ERR_SHAPE;
  if (n_item >= (int64_t(1) << 31) || n_vendor >= (int64_t(1) << 31) ||
      n_user >= (int64_t(1) << 31) || M >= (1 << 24) || K_user >= (1 << 24) ||
      K_vendor >= (1 << 24) || K_item >= (1 << 24))
    return IKBO_ERR_SHAPE;
  if (n_item == 0) return IKBO_OK;
  const bool has_u = K_user > 0, has_v = K_vendor > 0;
  if (!W_item || !X_item || !out || (has_u && (!W_user || !X_user || !vendor_to_user)) ||
      (has_v && (!W_vendor || !X_vendor)) || ((has_u || has_v) && !item_to_vendor))
    return IKBO_ERR_NULL;
  if ((has_u || has_v) && n_vendor == 0) return IKBO_ERR_INDEX;
  if (has_u && n_user == 0) return IKBO_ERR_INDEX;
  auto a4 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 3u) == 0; };
  if (!aligned16(W_item) || !aligned16(X_item) || !aligned16(out) ||
      (has_u && (!aligned16(W_user) || !aligned16(X_user) || !a4(vendor_to_user))) ||
      (has_v && (!aligned16(W_vendor) || !aligned16(X_vendor))) ||
      ((has_u || has_v) && !a4(item_to_vendor)))
    return IKBO_ERR_ALIGN;
  {
    const uintptr_t ob = reinterpret_cast<uintptr_t>(out), oe = ob + uintptr_t(n_item) * M * N * 2;
    auto overlaps = [&](bool used, const void* x, uintptr_t bytes) {
      const uintptr_t xb = reinterpret_cast<uintptr_t>(x);
      return used && x && xb < oe && ob < xb + bytes;
    };
    if (overlaps(true, W_item, uintptr_t(M) * K_item * 2) ||
        overlaps(true, X_item, uintptr_t(n_item) * K_item * N * 2) ||
        overlaps(has_u, W_user, uintptr_t(M) * K_user * 2) ||
        overlaps(has_u, X_user, uintptr_t(n_user) * K_user * N * 2) ||
        overlaps(has_v, W_vendor, uintptr_t(M) * K_vendor * 2) ||
        overlaps(has_v, X_vendor, uintptr_t(n_vendor) * K_vendor * N * 2) ||
        overlaps(has_u || has_v, item_to_vendor, uintptr_t(n_item) * 4) ||
        overlaps(has_u, vendor_to_user, uintptr_t(n_vendor) * 4))
      return IKBO_ERR_ALIAS;
  }
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int NB = N / 64;
  CUtensorMap wi_map, xi_map, wv_map, xv_map, wu_map, xu_map;
  std::memset(&wv_map, 0, sizeof wv_map);
  std::memset(&xv_map, 0, sizeof xv_map);
  std::memset(&wu_map, 0, sizeof wu_map);
  std::memset(&xu_map, 0, sizeof xu_map);
  if (encode_lce_w_map(&wi_map, W_item, M, K_item) != IKBO_OK ||
      encode_lce_x_map(&xi_map, X_item, n_item, K_item, N) != IKBO_OK ||
      (has_v && (encode_lce_w_map(&wv_map, W_vendor, M, K_vendor) != IKBO_OK ||
                 encode_lce_x_map(&xv_map, X_vendor, n_vendor, K_vendor, N) != IKBO_OK)) ||
      (has_u && (encode_lce_w_map(&wu_map, W_user, M, K_user) != IKBO_OK ||
                 encode_lce_x_map(&xu_map, X_user, n_user, K_user, N) != IKBO_OK)))
    return IKBO_ERR_CUDA;
  // bf16 terms of the user and vendor levels, library-owned, freed in stream order
  uint16_t* Yu = nullptr;
  uint16_t* Yv = nullptr;
  if (has_u && pool_alloc(ds, &Yu, size_t(n_user) * M * N * 2, st) !=
                   cudaSuccess)
    return IKBO_ERR_CUDA;
  if (has_v && pool_alloc(ds, &Yv, size_t(n_vendor) * M * N * 2, st) !=
                   cudaSuccess) {
    if (Yu) cudaFreeAsync(Yu, st);
    return IKBO_ERR_CUDA;
  }
  LceParams lp = {};
  lp.M = M;
  lp.N = N;
  lp.err_word = error_word(ds, st);
  lp.timeout_ns = g_timeout_ns;
  lp.cluster_n = lce_cluster_n(M, NB);
  cudaError_t e = cudaSuccess;
  if (g_timing) cudaEventRecord(ds->ev[0], st);
  if (has_u) {
    // users: Y_user[u] = W_user @ X_user[u]
    LceParams l = lp;
    l.W = static_cast<const uint16_t*>(W_user);
    l.n_batch = n_user;
    l.K = K_user;
    l.out = Yu;
    l.has_dependent = 1;
    e = launch_lce_nb(ds, NB, l, wu_map, xu_map, false, st);
  }
  if (g_timing) cudaEventRecord(ds->ev[1], st);
  if (e == cudaSuccess && has_v) {
    // vendors: Y_vendor[v] = W_vendor @ X_vendor[v] + Y_user[vendor_to_user[v]]
    LceParams l = lp;
    l.W = static_cast<const uint16_t*>(W_vendor);
    l.n_batch = n_vendor;
    l.K = K_vendor;
    l.out = Yv;
    l.has_dependent = 1;
    if (has_u) {
      l.add = 1;
      l.map = vendor_to_user;
      l.n_map = n_user;
      l.Y = Yu;
    }
    e = launch_lce_nb(ds, NB, l, wv_map, xv_map, has_u, st);
  }
  if (e == cudaSuccess) {
    // items: out[i] = W_item @ X_item[i] + the terms above, through item_to_vendor
    LceParams l = lp;
    l.W = static_cast<const uint16_t*>(W_item);
    l.n_batch = n_item;
    l.K = K_item;
    l.out = static_cast<uint16_t*>(out);
    if (has_u || has_v) {
      l.add = 1;
      l.map = item_to_vendor;
      l.n_map = n_vendor;
      l.Y = has_v ? Yv : Yu;
      if (has_u) {
        // with a vendor block, vendor_to_user is only checked here (the vendor
        // level has added the user term); without one, it finds the user's row
        l.map2 = vendor_to_user;
        l.n_map2 = n_user;
        l.y_via_map2 = has_v ? 0 : 1;
      }
    }
    e = launch_lce_nb(ds, NB, l, wi_map, xi_map, has_u || has_v, st);
  }
  if (g_timing) {
    cudaEventRecord(ds->ev[2], st);
    int dev = 0;
    cudaGetDevice(&dev);
    g_timing_dev = dev;
  }
  if (Yv) cudaFreeAsync(Yv, st);
  if (Yu) cudaFreeAsync(Yu, st);
  return e == cudaSuccess ? IKBO_OK : cuda_fail(e);
}

int ikbo_get_device_error(ikbo_stream_t stream) {
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != IKBO_OK) return rc;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return IKBO_ERR_CUDA;
  const size_t at = sizeof(int) * size_t(error_slot(ds, st, false));
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_ikbo_error_word, sizeof word, at) != cudaSuccess)
    return IKBO_ERR_CUDA;
  const int zero = 0;
  if (word && cudaMemcpyToSymbol(g_ikbo_error_word, &zero, sizeof zero, at) != cudaSuccess)
    return IKBO_ERR_CUDA;
  return status_of_error_word(word);
}

int ikbo_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  bool any = false;
  for (const DeviceState& s : g_dev) any = any || s.ready;
  if (!any) return IKBO_OK;   // nothing set up: no CUDA call at all
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return IKBO_ERR_CUDA;
  int rc = IKBO_OK;
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& s = g_dev[d];
    if (!s.ready) continue;
    if (cudaSetDevice(d) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) rc = IKBO_ERR_CUDA;
    // the streams' words start clean for whichever streams call next
    static const int zeros[kErrSlots] = {};
    if (cudaMemcpyToSymbol(g_ikbo_error_word, zeros, sizeof zeros) != cudaSuccess) rc = IKBO_ERR_CUDA;
    for (auto& e : s.ev)
      if (e) cudaEventDestroy(e);
    if (s.err_host) cudaFreeHost(s.err_host);
    delete s.host_call;
    delete s.calls;
    if (s.pool && (cudaMemPoolTrimTo(s.pool, 0) != cudaSuccess || cudaMemPoolDestroy(s.pool) != cudaSuccess))
      rc = IKBO_ERR_CUDA;
    s = DeviceState{};
  }
  g_timing_dev = -1;
  if (cudaSetDevice(prev) != cudaSuccess) rc = IKBO_ERR_CUDA;
  return rc;
}

const char* ikbo_strerror(int status) {
  switch (status) {
    case IKBO_OK: return "ok";
    case IKBO_ERR_NULL: return "a required pointer is NULL";
    case IKBO_ERR_SHAPE: return "unsupported shape (D must be 64 or 128, 1 <= Lq <= 128, H >= 1)";
    case IKBO_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case IKBO_ERR_SCALE: return "scale is not finite";
    case IKBO_ERR_CUDA: return "a CUDA call failed";
    case IKBO_ERR_INDEX: return "cand_to_user has a value outside [0, n_user)";
    case IKBO_ERR_OFFSETS: return "user_offsets is not a jagged index (offsets[0] != 0 or decreasing)";
    case IKBO_ERR_TIMEOUT: return "a bounded wait on the GPU ran out";
    case IKBO_ERR_ALIAS: return "out overlaps an input";
    case IKBO_ERR_DEVICE: return "the current device is not a compute capability 10.3 GPU";
    case IKBO_ERR_BUDGET: return "memory budget too small for one candidate's K/V copy";
    case IKBO_ERR_SCRATCH:
      return "the call needs more scratch than ikbo_attn_fwd_noalloc's fixed 40 MiB array";
    default: return "unknown status";
  }
}

int ikbo_version(void) { return kVersion; }

int ikbo_set_timing(int enable) {
  g_timing = enable != 0;
  return IKBO_OK;
}

int ikbo_get_timing(float* plan_ms, float* attn_ms) {
  if (g_timing_dev < 0) return IKBO_ERR_CUDA;
  DeviceState& s = g_dev[g_timing_dev];
  if (!s.ev_ready) return IKBO_ERR_CUDA;
  if (cudaEventSynchronize(s.ev[2]) != cudaSuccess) return IKBO_ERR_CUDA;
  float a = 0.f, b = 0.f;
  if (cudaEventElapsedTime(&a, s.ev[0], s.ev[1]) != cudaSuccess ||
      cudaEventElapsedTime(&b, s.ev[1], s.ev[2]) != cudaSuccess)
    return IKBO_ERR_CUDA;
  if (plan_ms) *plan_ms = a;
  if (attn_ms) *attn_ms = b;
  return IKBO_OK;
}

int ikbo_set_debug(int flags, uint64_t timeout_ns) {
  g_debug_flags = flags;
  g_timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
  return IKBO_OK;
}

int ikbo_pool_usage(int reset, uint64_t* used_now, uint64_t* used_high) {
  if (used_now) *used_now = 0;
  if (used_high) *used_high = 0;
  DeviceState* ds = nullptr;
  const int rc = device_state(&ds);
  if (rc != IKBO_OK) return rc;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    pool = ds->pool;
  }
  if (!pool) return IKBO_OK;
  uint64_t now = 0, high = 0;
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemCurrent, &now) != cudaSuccess ||
      cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &high) != cudaSuccess)
    return IKBO_ERR_CUDA;
  if (used_now) *used_now = now;
  if (used_high) *used_high = high;
  if (reset) {
    uint64_t zero = 0;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess)
      return IKBO_ERR_CUDA;
  }
  return IKBO_OK;
}

int ikbo_set_trace(uint64_t* device_buffer) {
  g_trace = device_buffer;
  return IKBO_OK;
}

int ikbo_set_kernel(int which) {
  const int prev = t_kernel;
  t_kernel = (which >= kKernAuto && which <= kKernAb) ? which : kKernAuto;
  return prev;
}

int ikbo_selected_kernel(int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq, int32_t D,
                         int64_t self_rows) {
  if (n_cand < 0 || n_user < 0 || H < 1 || Lq < 1 || Lq > kTileM || (D != 64 && D != 128))
    return IKBO_ERR_SHAPE;
  return effective_kernel(n_cand, n_user, H, Lq, D, self_rows < 0 ? -1 : self_rows);
}

int ikbo_launches_per_call(int64_t n_cand, int64_t n_user) {
  if (n_cand < 0 || n_user < 0) return IKBO_ERR_SHAPE;
  if (n_cand == 0) return 0;
  return (t_kernel != kKernSimt && fits_in_kernel_planning(n_cand, n_user)) ? 1 : 2;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of ikbo_attn_fwd.
//
// For callers that must not see the library allocate device memory (a memory
// manager that owns the whole device, or no stream-ordered pools), the
// scratch of the planning and attention kernels lives in this fixed array
// instead of the pool.  Host code only ever passes its device address, which
// is looked up once per device; the array's host-side name is a stand-in, not
// a device pointer.  Concurrent calls on the same device share it and race.
namespace ikbo {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[IKBO_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
char* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call there, with that device current).
int noalloc_scratch(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return IKBO_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return IKBO_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return IKBO_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<char*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return IKBO_OK;
}

}  // namespace
}  // namespace ikbo

extern "C" int ikbo_attn_fwd_noalloc(const void* q, const void* k_user, const void* v_user,
                                     const int32_t* user_offsets, const int32_t* cand_to_user,
                                     int64_t n_cand, int64_t n_user, int32_t H, int32_t Lq,
                                     int32_t D, float scale, void* out, ikbo_stream_t stream) {
  using namespace ikbo;
  int rc = check_args(q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                      scale, out);
  if (rc != IKBO_OK || n_cand == 0) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != IKBO_OK) return rc;
  if (g_timing && (rc = ensure_events(ds)) != IKBO_OK) return rc;
  Workspace L;
  if ((rc = call_workspace(ds, n_cand, n_user, H, Lq, D, &L)) != IKBO_OK) return rc;
  if (L.total > size_t(IKBO_NOALLOC_SCRATCH_BYTES)) return IKBO_ERR_SCRATCH;
  char* ws = nullptr;
  if ((rc = noalloc_scratch(&ws)) != IKBO_OK) return rc;
  return run_ikbo(ds, q, k_user, v_user, user_offsets, cand_to_user, n_cand, n_user, H, Lq, D,
                  scale, out, ws, L, reinterpret_cast<cudaStream_t>(stream));
}

