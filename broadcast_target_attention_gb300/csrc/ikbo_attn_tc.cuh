// IKBO target attention on the 5th-generation tensor cores (sm_103a):
// persistent, warp-specialised, TMA-fed, accumulators in tensor memory,
// launched as clusters of two CTAs.
//
// What it computes: for every work item (one user, one head, a query tile of
// up to 128 rows = that user's candidates x Lq tokens, one range of the
// user's keys) the flash-attention forward of "Chapter 4: High-performance
// Kernels", §4.6.1: S = Q K^T tile by tile, online softmax (running max m,
// running sum l, rescaled output), O += P V, out = O / l.
//
// Where IKBO enters ("In-Kernel Broadcast Optimization", §3.1-§3.2): the
// rows of a query tile are the queries of several candidates of ONE user, so
// every K/V tile that the TMA brings into shared memory serves all of them;
// the user's sequence is found through user_offsets, never through a
// per-candidate copy.  A tile that is only partly filled (odd or short
// groups, §3.2 "generalised" kernel) simply carries unused rows: the MMA
// computes them, the epilogue does not store them, and no warp waits for a
// partner that does not exist.
//
// Planning.  For inputs of moderate size every CTA plans in its prologue,
// from the index tensors, with its shared memory as scratch: it validates
// cand_to_user and user_offsets, groups candidates by user (a stable counting
// sort when the map is unsorted), orders users longest first and derives its
// own work items, so the whole forward is ONE launch.  Larger inputs use the
// separate planning kernel's work list.  Items are handed to CTAs in
// boustrophedon order over the longest-first list ("Optimizing Jagged Flash
// Attention with TLX", §2.2: tiles sorted by K/V work, even passes left to
// right, odd passes right to left); the items of one (user, head) are
// adjacent so CTAs sharing a user's K/V run together ("In-Kernel Broadcast
// Optimization", §3.1, Table 1).
//
// Pair mode.  When there are no more (user, head, query tile) units than
// clusters, the two CTAs of a cluster split one unit's keys in half.  The
// second CTA sends its un-normalised O and (m, l) through distributed shared
// memory into the first, which merges them with the log-sum-exp rule of
// "Chapter 4", §4.6.4 (Flash-Decoding): M = max(m0, m1),
// out = (2^(m0-M) O0 + 2^(m1-M) O1) / (2^(m0-M) l0 + 2^(m1-M) l1).
//
// Warp roles (256 threads), after the Blackwell design of "Optimizing Jagged
// Flash Attention with TLX", §2.1 (dedicated load, MMA and softmax warps;
// explicit SMEM/TMEM buffers; S/P sharing one TMEM buffer, the PV
// accumulator its own; persistent CTAs):
//   warp 0      TMA producer: Q tile, then K_0, K_1, V_0, K_2, V_1, ... into a
//               ring of shared-memory slots;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T (SS form) into one of two S buffers, then
//               O += P_{j-1} V_{j-1} (TS form, P read from TMEM), so S_j
//               overlaps the softmax of tile j-1;
//   warps 4-7   softmax, O correction and epilogue; thread i owns TMEM lane
//               (= query row) i.
// Every wait is bounded: a wait that runs out sets the device error word,
// raises an abort flag that ends all roles, and the CTA drains its
// outstanding copies and MMAs before freeing tensor memory.
#pragma once

#include <cuda_bf16.h>

#include "ikbo_common.cuh"
#include "ikbo_ptx.cuh"

namespace ikbo {

constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kTcThreads = 256;
// The running maximum is moved only when a tile's maximum exceeds it by more
// than this (base-2 units), so un-normalised weights stay <= 2^8 and the
// O correction is skipped on most tiles; the final O / l is exact either way.
constexpr float kLazyRescale = 8.0f;
constexpr int kDataBytes = 229376;   // 224 KB: operands (and planning scratch in the prologue)
constexpr int kCtrlBytes = 2048;     // barriers, flags, plan results, partner (m, l)
constexpr int kTcSmemBytes = kCtrlBytes + 1024 + kDataBytes;   // = 227 KB, the per-CTA maximum
constexpr int kMaxSlots = 14;
// In-kernel planning keeps off/cand_start/order/prefix (n_user), the per-warp
// counters of the counting sort (8 x n_user) and cand_to_user/perm (n_cand)
// in the operand area.
constexpr int kFusedMaxUser = 1024;
constexpr int kFusedMaxCand = 20480;
constexpr int kLptMaxUsersFused = 256;

enum TcMode { kModeSkip = -1, kModeListed = 0, kModeIndep = 1, kModePair = 2 };
constexpr int kCtlItems = 4;

template <int D>
struct TcConfig {
  static constexpr int kCB = D / 64;                   // 128-byte column blocks per row
  static constexpr int kQBytes = kCB * kTileM * 128;    // one Q tile
  static constexpr int kKVBytes = kCB * kBlockN * 128;  // one K or V tile
  // Operand area: two Q buffers, then the K/V ring.  In pair mode only the
  // first Q buffer is used and both together receive the partner's O.
  static constexpr int kSlots = (kDataBytes - 2 * kQBytes) / kKVBytes;
  static constexpr int kRecvBytes = kTileM * D * 4;
  // tensor-memory columns: two S/P buffers and the O accumulator
  static constexpr int kSCol = 0;
  static constexpr int kOCol = 2 * kBlockN;
  static constexpr int kTmemCols = 512;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static_assert(kSlots <= kMaxSlots && kSlots >= 3, "ring size");
  static_assert(kRecvBytes == 2 * kQBytes, "receive area = both Q buffers");
  static_assert(kRecvBytes + 16 * kTileM <= kSlots * kKVBytes, "staging area");
};

static_assert(kTcSmemBytes <= 232448, "shared memory budget");
static_assert(4 * (4 * (kFusedMaxUser + 1) + 8 * kFusedMaxUser + 2 * kFusedMaxCand) <= kDataBytes,
              "planning scratch");

// Control block at the start of dynamic shared memory.
struct TcCtrl {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, drain, pair_go, pair_recv, stage_done;
  uint32_t tmem_base;
  int abort_flag;
  int wg_count;
  int mode;
  int n_my_items;
  int sorted;
  int n_slots;
  int go_sent;
  int red_i[32];
  WorkItem items[kCtlItems];            // the first items of this CTA (the rest in global memory)
  alignas(16) float2 partner_ml[kTileM];
};
static_assert(sizeof(TcCtrl) <= kCtrlBytes, "control block");

// Bounded mbarrier wait shared by all roles of a CTA.
struct Waiter {
  volatile int* abort;
  int* err_word;
  uint64_t timeout_ns;

  __device__ __forceinline__ bool poll(uint32_t bar, uint32_t parity, bool cluster) const {
    return cluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  }
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, bool cluster = false) const {
    if (poll(bar, parity, cluster)) return true;
    uint64_t t_end = 0;
    for (uint32_t spin = 1;; ++spin) {
      if (*abort) return false;
      if (poll(bar, parity, cluster)) return true;
      if ((spin & 63u) == 0) {
        const uint64_t now = ptx::globaltimer();
        if (t_end == 0) {
          t_end = now + timeout_ns;
        } else if (now > t_end) {
          *abort = 1;
          atomicOr(err_word, kErrTimeout);
          return false;
        }
      }
    }
  }
  // Drain waits ignore the abort flag (they only wait for work already issued)
  // but are bounded all the same.
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    uint64_t t_end = 0;
    for (uint32_t spin = 0;; ++spin) {
      if (ptx::mbar_try_wait(bar, parity)) return true;
      if ((spin & 63u) == 63u) {
        const uint64_t now = ptx::globaltimer();
        if (t_end == 0) {
          t_end = now + timeout_ns;
        } else if (now > t_end) {
          atomicOr(err_word, kErrTimeout);
          return false;
        }
      }
    }
  }
  // One lane polls, the warp follows its verdict.
  __device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, bool cluster = false) const {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait(bar, parity, cluster) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
  }
};

__device__ __forceinline__ void trace(const AttnParams& p, int ord, int point) {
  if (p.trace && ord < kTraceItems)
    p.trace[(size_t(blockIdx.x) * kTraceItems + ord) * kTracePoints + point] = ptx::globaltimer();
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Block-wide exclusive scan of one int per thread (all threads call it).
__device__ __forceinline__ int block_scan_excl(int x, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    red[lane] = w;
  }
  __syncthreads();
  const int pre = warp == 0 ? 0 : red[warp - 1];
  *total = red[nw - 1];
  __syncthreads();
  return pre + v - x;
}

// ---------------------------------------------------------------------------
// In-kernel planning.  All threads of the CTA; `scratch` is the operand area.
// Every CTA computes the same plan (the inputs are small) and keeps only its
// own items.  The K/V tensor maps get their row count T here, in a per-CTA
// slot in global memory.
// ---------------------------------------------------------------------------
__device__ void plan_in_cta(const AttnParams& p, TcCtrl* ctl, uint8_t* scratch,
                            const CUtensorMap& kt, const CUtensorMap& vt, int D) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int grid = gridDim.x, b = blockIdx.x;
  const int n_cand = (int)p.n_cand, n_user = (int)p.n_user;
  int32_t* off = reinterpret_cast<int32_t*>(scratch);   // n_user + 1
  int32_t* cs = off + (n_user + 1);                     // cand_start, n_user + 1
  int32_t* order = cs + (n_user + 1);                   // n_user
  int32_t* ubefore = order + n_user;                    // n_user + 1
  int32_t* wcnt = ubefore + (n_user + 1);               // 8 x n_user (unsorted only)
  int32_t* c2u = wcnt + 8 * n_user;                     // n_cand
  int32_t* perm = c2u + n_cand;                         // n_cand

  for (int u = tid; u <= n_user; u += nt) off[u] = p.user_offsets[u];
  for (int c = tid; c < n_cand; c += nt) c2u[c] = p.cand_to_user[c];
  __syncthreads();
  // K/V tensor maps: row count T, into this CTA's global slots
  if (tid == 0) {
    const int T = off[n_user];
    const int rows = T > 0 ? T : 1;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      CUtensorMap* dst = p.map_slots + 2 * b + mi;
      const uint4* s4 = reinterpret_cast<const uint4*>(mi == 0 ? &kt : &vt);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
      asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(dst),
                   "r"(rows)
                   : "memory");
    }
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
  // validation
  int e_off = 0, e_idx = 0, unsorted = 0;
  if (tid == 0 && off[0] != 0) e_off = 1;
  for (int u = tid; u < n_user; u += nt)
    if (off[u + 1] < off[u]) e_off = 1;
  for (int c = tid; c < n_cand; c += nt) {
    const int x = c2u[c];
    if (x < 0 || x >= n_user) e_idx = 1;
    if (c > 0 && c2u[c - 1] > x) unsorted = 1;
  }
  const int any_off = __syncthreads_or(e_off);
  const int any_idx = __syncthreads_or(e_idx);
  const int any_uns = __syncthreads_or(unsorted);
  if (any_off || any_idx) {
    if (tid == 0) {
      ctl->mode = kModeSkip;
      ctl->n_my_items = 0;
      ctl->sorted = 1;
      if (b == 0) atomicOr(p.err_word, (any_off ? kErrOffsets : 0) | (any_idx ? kErrIndex : 0));
    }
    __syncthreads();
    return;
  }
  // group candidates by user
  if (!any_uns) {
    for (int c = tid; c < n_cand; c += nt) {
      const int x = c2u[c];
      const int prev = c == 0 ? -1 : c2u[c - 1];
      for (int uu = prev + 1; uu <= x; ++uu) cs[uu] = c;
    }
    for (int uu = c2u[n_cand - 1] + 1 + tid; uu <= n_user; uu += nt) cs[uu] = n_cand;
    __syncthreads();
  } else {
    // stable counting sort: warp w owns a contiguous segment of candidates
    const int warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
    const int seg = (n_cand + nw - 1) / nw;
    const int seg_end = min(n_cand, (warp + 1) * seg);
    for (int i = tid; i < nw * n_user; i += nt) wcnt[i] = 0;
    __syncthreads();
    for (int c = warp * seg + lane; c < seg_end; c += 32) atomicAdd(&wcnt[warp * n_user + c2u[c]], 1);
    __syncthreads();
    // per-user totals -> cand_start (exclusive scan over users)
    int carry = 0;
    for (int base = 0; base < n_user; base += nt) {
      const int u = base + tid;
      int tot_u = 0;
      if (u < n_user)
        for (int w = 0; w < nw; ++w) tot_u += wcnt[w * n_user + u];
      int tot;
      const int ex = block_scan_excl(tot_u, ctl->red_i, &tot);
      if (u < n_user) cs[u] = carry + ex;
      carry += tot;
    }
    if (tid == 0) cs[n_user] = n_cand;
    __syncthreads();
    // per-warp cursors: cand_start + counts of the earlier warps
    for (int u = tid; u < n_user; u += nt) {
      int acc = cs[u];
      for (int w = 0; w < nw; ++w) {
        const int cnt = wcnt[w * n_user + u];
        wcnt[w * n_user + u] = acc;
        acc += cnt;
      }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = warp * seg; base < seg_end; base += 32) {
      const int c = base + lane;
      const bool valid = c < seg_end;
      const int x = valid ? c2u[c] : -1;
      const unsigned same = __match_any_sync(0xffffffffu, x);
      int pos = 0;
      if (valid) pos = wcnt[warp * n_user + x] + __popc(same & lt);
      __syncwarp();
      if (valid && (same & lt) == 0) wcnt[warp * n_user + x] += __popc(same);
      if (valid) perm[pos] = c;
      __syncwarp();
    }
    __syncthreads();
    // every CTA writes the same permutation; each reads back only its own writes
    for (int i = tid; i < n_cand; i += nt) p.perm_ws[i] = perm[i];
  }
  // rows of candidates whose user has an empty sequence are zero
  {
    const int64_t elems = (int64_t)p.H * p.Lq * D;
    for (int c = b * nt + tid; c < n_cand; c += grid * nt) {
      const int x = c2u[c];
      if (off[x + 1] == off[x]) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)c * elems);
        for (int64_t i = 0; i < elems / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  // users, longest first (index order beyond kLptMaxUsersFused users)
  for (int u = tid; u < n_user; u += nt) {
    if (n_user <= kLptMaxUsersFused) {
      const int Lu = off[u + 1] - off[u];
      int rank = 0;
      for (int w = 0; w < n_user; ++w) {
        const int Lw = off[w + 1] - off[w];
        rank += (Lw > Lu) || (Lw == Lu && w < u);
      }
      order[rank] = u;
    } else {
      order[u] = u;
    }
  }
  __syncthreads();
  // units per rank: H x query tiles of users with candidates and keys
  const int cpt = p.cands_per_tile;
  {
    int carry = 0;
    for (int base = 0; base < n_user; base += nt) {
      const int rk = base + tid;
      int nu = 0;
      if (rk < n_user) {
        const int u = order[rk];
        const int r = cs[u + 1] - cs[u], L = off[u + 1] - off[u];
        if (r > 0 && L > 0) nu = p.H * ceil_div(r, cpt);
      }
      int tot;
      const int ex = block_scan_excl(nu, ctl->red_i, &tot);
      if (rk < n_user) ubefore[rk] = carry + ex;
      carry += tot;
    }
    if (tid == 0) ubefore[n_user] = carry;
    __syncthreads();
  }
  const int N = ubefore[n_user];
  const bool pair = N > 0 && 2 * N <= grid;
  // decode unit i into a work item
  auto decode = [&](int i, WorkItem& w) {
    int lo = 0, hi = n_user - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ubefore[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int u = order[lo];
    const int r = cs[u + 1] - cs[u];
    const int nmt = ceil_div(r, cpt);
    const int local = i - ubefore[lo];
    const int h = local / nmt, mt = local - h * nmt;
    w.user = u;
    w.head = h;
    w.cand_begin = cs[u] + mt * cpt;
    w.n_cand = min(cpt, r - mt * cpt);
    w.kv_begin = off[u];
    w.kv_len = off[u + 1] - off[u];
    w.unit = -1;
    w.unit_first = 0;
  };
  WorkItem* mine = p.cta_items + (size_t)b * p.max_cta_items;
  if (pair) {
    if (tid == 0) {
      const int c = b >> 1, rank = b & 1;
      int count = 0;
      if (c < N) {
        WorkItem w;
        decode(c, w);
        const int kt = ceil_div(w.kv_len, kBlockN);
        if (kt >= 2) {
          const int first = ceil_div(kt, 2) * kBlockN;   // keys of the leader
          if (rank == 0) {
            w.kv_len = first;
            w.unit = 0;
            w.unit_first = 1;
          } else {
            w.kv_begin += first;
            w.kv_len -= first;
            w.unit = 1;
          }
          mine[0] = w;
          ctl->items[0] = w;
          count = 1;
        } else if (rank == 0) {
          mine[0] = w;
          ctl->items[0] = w;
          count = 1;
        }
      }
      ctl->n_my_items = count;
    }
  } else {
    const int full = N / grid, rem = N - full * grid;
    const int pos_last = (full & 1) ? grid - 1 - b : b;
    int count = full + (pos_last < rem ? 1 : 0);
    count = min(count, p.max_cta_items);
    for (int k = tid; k < count; k += nt) {
      const int i = k * grid + ((k & 1) ? grid - 1 - b : b);
      WorkItem w;
      decode(i, w);
      mine[k] = w;
      if (k < kCtlItems) ctl->items[k] = w;
    }
    if (tid == 0) ctl->n_my_items = count;
  }
  if (tid == 0) {
    ctl->mode = pair ? kModePair : kModeIndep;
    ctl->sorted = any_uns ? 0 : 1;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
ikbo_attn_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap qmap1,
                    const __grid_constant__ CUtensorMap kmap_tmpl,
                    const __grid_constant__ CUtensorMap vmap_tmpl) {
  using C = TcConfig<D>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem_raw);
  uint8_t* data = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + kCtrlBytes + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta_rank = ptx::cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->q_empty[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[i]), 4);
    }
    for (int i = 0; i < kMaxSlots; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->pv_done), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_go), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_recv), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->stage_done), 4);
    ctl->go_sent = 0;
    ctl->abort_flag = 0;
    ctl->wg_count = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // A planning kernel may precede this one (programmatic dependent launch):
  // its work list is visible after this wait.  Without one it returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.fused) {
    __syncthreads();
    plan_in_cta(p, ctl, data, kmap_tmpl, vmap_tmpl, D);
    // the planning scratch is overwritten by TMA (async proxy) from here on
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  } else if (threadIdx.x == 0) {
    ctl->mode = kModeListed;
    ctl->sorted = p.header->sorted != 0;
    const int n = p.header->n_items;
    ctl->n_my_items =
        n > (int)blockIdx.x ? (n - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  }
  if (threadIdx.x == 0) {
    ctl->n_slots = C::kSlots;
    trace(p, 0, kTrCtaStart);
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the partner's barriers are initialised before any remote arrive
  ptx::cluster_sync();
  ptx::tc_fence_after();

  const uint32_t tmem = ctl->tmem_base;
  const int mode = ctl->mode;
  const int n_my = ctl->n_my_items;
  const bool sorted = ctl->sorted != 0;
  const int NS = ctl->n_slots;
  const int NQ = mode == kModePair ? 1 : 2;
  uint8_t* q_smem = data;
  uint8_t* kv_smem = data + 2 * C::kQBytes;
  const int32_t* perm = p.fused ? p.perm_ws : p.perm;
  const void* kmap = p.fused ? (const void*)(p.map_slots + 2 * blockIdx.x) : p.kmap;
  const void* vmap = p.fused ? (const void*)(p.map_slots + 2 * blockIdx.x + 1) : p.vmap;
  const Waiter W{&ctl->abort_flag, p.err_word, p.timeout_ns};
  const int Lq = p.Lq;
  auto item_at = [&](int k) -> WorkItem {
    if (p.fused) return k < kCtlItems ? ctl->items[k] : p.cta_items[(size_t)blockIdx.x * p.max_cta_items + k];
    return p.items[blockIdx.x + (size_t)k * gridDim.x];
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && mode != kModeSkip) {
      ptx::tensormap_acquire(kmap);
      ptx::tensormap_acquire(vmap);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      auto load_tile = [&](const void* map, int head, int32_t row) -> bool {
        const uint32_t slot = kv_it % NS;
        if (!W.wait(ptx::smem_addr(&ctl->kv_empty[slot]), ((kv_it / NS) & 1u) ^ 1u)) return false;
        const uint32_t bar = ptx::smem_addr(&ctl->kv_full[slot]);
        const uint32_t dst = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
        ptx::mbar_arrive_expect_tx(bar, C::kKVBytes);
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb)
          ptx::tma_load_2d(dst + cb * kBlockN * 128, map, bar, head * D + cb * 64, row);
        ++kv_it;
        return true;
      };
      for (int k = 0; k < n_my && ok; ++k) {
        const WorkItem w = item_at(k);
        const int n = ceil_div(w.kv_len, kBlockN);
        const uint32_t qb = q_it % NQ;
        const uint32_t qpar = ((q_it / NQ) & 1u) ^ 1u;
        trace(p, k, kTrProdItem);
        if (!W.wait(ptx::smem_addr(&ctl->q_empty[qb]), qpar)) break;
        const uint32_t qbar = ptx::smem_addr(&ctl->q_full[qb]);
        const uint32_t qdst = ptx::smem_addr(q_smem + qb * C::kQBytes);
        if (!(p.debug_flags & 1)) {
          if (sorted) {
            const int nb = p.qbox;
            const int nbox = ceil_div(w.n_cand, nb);
            ptx::mbar_arrive_expect_tx(qbar, uint32_t(nbox * nb * Lq * 128 * C::kCB));
            for (int cb = 0; cb < C::kCB; ++cb)
              for (int bx = 0; bx < nbox; ++bx)
                ptx::tma_load_4d(qdst + cb * kTileM * 128 + bx * nb * Lq * 128, &qmap, qbar,
                                 cb * 64, 0, w.head, w.cand_begin + bx * nb);
          } else {
            ptx::mbar_arrive_expect_tx(qbar, uint32_t(w.n_cand * Lq * 128 * C::kCB));
            for (int i = 0; i < w.n_cand; ++i) {
              const int32_t c = perm[w.cand_begin + i];
              for (int cb = 0; cb < C::kCB; ++cb)
                ptx::tma_load_4d(qdst + cb * kTileM * 128 + i * Lq * 128, &qmap1, qbar, cb * 64, 0,
                                 w.head, c);
            }
          }
        }
        ++q_it;
        // K/V tiles in the order the MMA warp consumes them: K0, K1, V0, K2, V1, ...
        for (int j = 0; j <= n && ok; ++j) {
          if (j < n) ok = load_tile(kmap, w.head, w.kv_begin + j * kBlockN);
          if (ok && j >= 1) ok = load_tile(vmap, w.head, w.kv_begin + (j - 1) * kBlockN);
        }
        trace(p, k, kTrProdIssued);
        if (ok && w.unit == 0 && w.unit_first) {
          // pair leader: once the last S has read Q, both Q buffers can receive
          // the partner's O and (m, l); tell the partner so
          if (!W.wait(ptx::smem_addr(&ctl->q_empty[0]), 0)) break;
          const int rows = w.n_cand * Lq;
          const uint32_t bytes = uint32_t(rows * D * 4 + ((rows + 1) & ~1) * 8);
          ptx::mbar_arrive_expect_tx(ptx::smem_addr(&ctl->pair_recv), bytes);
          ctl->go_sent = 1;
          ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_addr(&ctl->pair_go), cta_rank ^ 1u));
        }
      }
      // Drain: every armed barrier phase must complete before the CTA exits.
      for (uint32_t s = 0; s < (uint32_t)NS && s < kv_it; ++s) {
        const uint32_t uses = (kv_it - s + NS - 1) / NS;
        W.drain(ptx::smem_addr(&ctl->kv_full[s]), (uses - 1) & 1u);
      }
      if (!(p.debug_flags & 1))
        for (uint32_t qb = 0; qb < (uint32_t)NQ && qb < q_it; ++qb) {
          const uint32_t uses = (q_it - qb + NQ - 1) / NQ;
          W.drain(ptx::smem_addr(&ctl->q_full[qb]), (uses - 1) & 1u);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0 && mode != kModeSkip) {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kTileM, kBlockN, 0);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kTileM, 64, 1);
      uint32_t kv_it = 0, q_it = 0, g = 0;
      bool ok = true;
      for (int k = 0; k < n_my && ok; ++k) {
        const WorkItem w = item_at(k);
        const int n = ceil_div(w.kv_len, kBlockN);
        const uint32_t qb = q_it % NQ;
        if (!W.wait(ptx::smem_addr(&ctl->q_full[qb]), (q_it / NQ) & 1u)) break;
        ptx::tc_fence_after();
        trace(p, k, kTrMmaQ);
        const uint32_t q_base = ptx::smem_addr(q_smem + qb * C::kQBytes);
        for (int j = 0; j <= n; ++j) {
          if (j < n) {
            const uint32_t slot = kv_it % NS;
            if (!W.wait(ptx::smem_addr(&ctl->kv_full[slot]), (kv_it / NS) & 1u)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t k_base = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
            const uint32_t sb = (g + j) & 1u;
            const uint32_t d_tmem = tmem + C::kSCol + sb * kBlockN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int cb = kk >> 2;
              const uint32_t koff = (kk & 3) * 32;
              const uint64_t a = ptx::smem_desc_sw128(q_base + cb * kTileM * 128 + koff, 16, 1024);
              const uint64_t bdesc = ptx::smem_desc_sw128(k_base + cb * kBlockN * 128 + koff, 16, 1024);
              ptx::mma_ss(d_tmem, a, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
            }
            if (j == 0) trace(p, k, kTrMmaFirstS);
            ptx::mma_commit(ptx::smem_addr(&ctl->kv_empty[slot]));
            ptx::mma_commit(ptx::smem_addr(&ctl->s_full[sb]));
            if (j == n - 1) ptx::mma_commit(ptx::smem_addr(&ctl->q_empty[qb]));
            ++kv_it;
          }
          if (j >= 1) {
            const uint32_t pj = g + j - 1;
            const uint32_t pb = pj & 1u;
            if (!W.wait(ptx::smem_addr(&ctl->p_full[pb]), (pj >> 1) & 1u)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t slot = kv_it % NS;
            if (!W.wait(ptx::smem_addr(&ctl->kv_full[slot]), (kv_it / NS) & 1u)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t v_base = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
            const uint32_t a_tmem = tmem + C::kSCol + pb * kBlockN;
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
#pragma unroll
              for (int cb = 0; cb < C::kCB; ++cb) {
                const uint64_t bdesc = ptx::smem_desc_sw128(
                    v_base + cb * kBlockN * 128 + kk * 16 * 128, kBlockN * 128, 1024);
                ptx::mma_ts(tmem + C::kOCol + cb * 64, a_tmem + kk * 8, bdesc, kIdescPV,
                            (j > 1 || kk > 0) ? 1u : 0u);
              }
            }
            ptx::mma_commit(ptx::smem_addr(&ctl->kv_empty[slot]));
            ptx::mma_commit(ptx::smem_addr(&ctl->pv_done));
            if (j == n) trace(p, k, kTrMmaLastPV);
            ++kv_it;
          }
        }
        g += n;
        ++q_it;
      }
      // All issued MMAs must finish before tensor memory is released.
      ptx::mma_commit(ptx::smem_addr(&ctl->drain));
      W.drain(ptx::smem_addr(&ctl->drain), 0);
    }
    __syncwarp();
  } else if (warp >= 4 && mode != kModeSkip) {
    // ------------------------------------------- softmax / correction / epilogue
    const int row = threadIdx.x - 128;                       // TMEM lane == tile row
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, pv_it = 0;
    for (int k = 0; k < n_my; ++k) {
      const WorkItem w = item_at(k);
      const int n = ceil_div(w.kv_len, kBlockN);
      const int rows = w.n_cand * Lq;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1u;
        if (!W.warp_wait(ptx::smem_addr(&ctl->s_full[sb]), (gj >> 1) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (j == 0 && row == 0) trace(p, k, kTrSmS0);
        const uint32_t scol = tmem + lane_off + C::kSCol + sb * kBlockN;
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(scol + c * 32, sr[c]);
        ptx::tmem_ld_wait();
        const int valid = min(kBlockN, w.kv_len - j * kBlockN);
        // row maximum of the scaled scores (of the raw minimum when scale < 0)
        const float sgn = sl2 < 0.f ? -1.f : 1.f;
        float mxv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxv[e] = -INFINITY;
        if (valid == kBlockN) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) mxv[e & 7] = fmaxf(mxv[e & 7], sgn * __uint_as_float(sr[c][e]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < valid) mxv[e & 7] = fmaxf(mxv[e & 7], sgn * __uint_as_float(sr[c][e]));
        }
        float mx = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                         fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
        mx *= sgn * sl2;
        const float m_new = (m == -INFINITY || mx > m + kLazyRescale) ? fmaxf(m, mx) : m;
        const float alpha = fast_exp2(m - m_new);   // 0 on the first tile, 1 when m stays
        float sumv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) sumv[e] = 0.f;
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = c * 32 + e;
            float p0 = fast_exp2(fmaf(__uint_as_float(sr[c][e]), sl2, -m_new));
            float p1 = fast_exp2(fmaf(__uint_as_float(sr[c][e + 1]), sl2, -m_new));
            if (valid < kBlockN) {
              p0 = col < valid ? p0 : 0.f;
              p1 = col + 1 < valid ? p1 : 0.f;
            }
            sumv[(e >> 1) & 7] += p0 + p1;
            pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16(p0, p1);
          }
        const float sum = ((sumv[0] + sumv[1]) + (sumv[2] + sumv[3])) +
                          ((sumv[4] + sumv[5]) + (sumv[6] + sumv[7]));
        l = l * alpha + sum;
        // P (bf16 pairs) overwrites the first half of this S buffer.
        ptx::tmem_st32(scol, pk[0]);
        ptx::tmem_st32(scol + 32, pk[1]);
        ptx::tmem_st_wait();
        if (j > 0) {
          // O holds P_0..P_{j-1} V: wait for PV_{j-1}, then rescale if m moved.
          if (!W.warp_wait(ptx::smem_addr(&ctl->pv_done), pv_it & 1u)) {
            ok = false;
            break;
          }
          ++pv_it;
          ptx::tc_fence_after();
          if (__any_sync(0xffffffffu, m_new != m)) {
            const uint32_t ocol = tmem + lane_off + C::kOCol;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              ptx::tmem_ld32(ocol + c * 32, o);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              ptx::tmem_st32(ocol + c * 32, o);
            }
            ptx::tmem_st_wait();
          }
        }
        m = m_new;
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl->p_full[sb]));
      }
      if (!ok) break;
      if (row == 0) trace(p, k, kTrSmLastP);
      // ---- epilogue
      if (!W.warp_wait(ptx::smem_addr(&ctl->pv_done), pv_it & 1u)) break;
      ++pv_it;
      ptx::tc_fence_after();
      if (row == 0) trace(p, k, kTrEpiO);
      const uint32_t ocol = tmem + lane_off + C::kOCol;
      const bool live = row < rows;
      const int ci = live ? row / Lq : 0;
      const int t = live ? row - ci * Lq : 0;
      if (w.unit == 1) {
        // pair sender: stage O (swizzled rows) and (m, l) in this CTA's ring,
        // which no MMA reads any more, then one bulk copy into the leader
        uint8_t* stage = kv_smem;
        float2* stage_ml = reinterpret_cast<float2*>(kv_smem + C::kRecvBytes);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + cc * 32, o);
          ptx::tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const int vec = cc * 8 + q4;                     // 16-byte vector of the row
              *reinterpret_cast<uint4*>(stage + row * (D * 4) + ((vec ^ (row & 7)) * 16)) =
                  make_uint4(o[q4 * 4 + 0], o[q4 * 4 + 1], o[q4 * 4 + 2], o[q4 * 4 + 3]);
            }
          }
        }
        if (live) stage_ml[row] = make_float2(m, l);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl->stage_done));
        if (row == 0) {
          if (W.wait(ptx::smem_addr(&ctl->stage_done), 0) &&
              W.wait(ptx::smem_addr(&ctl->pair_go), 0, true)) {
            const uint32_t peer = cta_rank ^ 1u;
            const uint32_t rbar = ptx::map_to_cta(ptx::smem_addr(&ctl->pair_recv), peer);
            ptx::bulk_copy_to_cta(ptx::map_to_cta(ptx::smem_addr(data), peer), ptx::smem_addr(stage),
                                  uint32_t(rows * D * 4), rbar);
            ptx::bulk_copy_to_cta(ptx::map_to_cta(ptx::smem_addr(ctl->partner_ml), peer),
                                  ptx::smem_addr(stage_ml), uint32_t(((rows + 1) & ~1) * 8), rbar);
            trace(p, k, kTrEpiStored);
          }
        }
        __syncwarp();
      } else {
        const int32_t gpos = w.cand_begin + ci;
        const int64_t cidx = live ? (sorted ? gpos : perm[gpos]) : 0;
        uint16_t* dst = p.out + (((cidx * p.H + w.head) * (int64_t)Lq + t) * D);
        float mp = -INFINITY, lp = 0.f;
        const bool merge = w.unit == 0 && w.unit_first != 0;
        if (merge) {
          // pair leader: the partner's O and (m, l) arrive in the Q buffers
          if (!W.warp_wait(ptx::smem_addr(&ctl->pair_recv), 0, true)) break;
          if (row == 0) trace(p, k, kTrArrived);
          if (live) {
            const float2 ml = ctl->partner_ml[row];
            mp = ml.x;
            lp = ml.y;
          }
        }
        const float M = fmaxf(m, mp);
        const float a0 = fast_exp2(m - M), a1 = merge ? fast_exp2(mp - M) : 0.f;
        const float L = a0 * l + a1 * lp;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + cc * 32, o);
          ptx::tmem_ld_wait();
          if (live) {
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(o[e]) * w0;
            if (merge) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const int vec = cc * 8 + q4;
                const float4 y = *reinterpret_cast<const float4*>(
                    data + row * (D * 4) + ((vec ^ (row & 7)) * 16));
                x[q4 * 4 + 0] += y.x * w1;
                x[q4 * 4 + 1] += y.y * w1;
                x[q4 * 4 + 2] += y.z * w1;
                x[q4 * 4 + 3] += y.w * w1;
              }
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = pack_bf16(x[q4 * 8 + 0], x[q4 * 8 + 1]);
              v.y = pack_bf16(x[q4 * 8 + 2], x[q4 * 8 + 3]);
              v.z = pack_bf16(x[q4 * 8 + 4], x[q4 * 8 + 5]);
              v.w = pack_bf16(x[q4 * 8 + 6], x[q4 * 8 + 7]);
              d4[q4] = v;
            }
          }
        }
        if (row == 0) trace(p, k, merge ? kTrMerged : kTrEpiStored);
      }
      g += n;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // a leader that invited its partner's copy waits for it (bounded) before
  // its shared memory can go away, even if it gave up on the merge
  if (threadIdx.x == 0 && ctl->go_sent) W.drain(ptx::smem_addr(&ctl->pair_recv), 0);
  if (threadIdx.x == 0) trace(p, 0, kTrCtaEnd);
  __syncwarp();
  // neither CTA of a pair may exit while the other can still touch its memory
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace ikbo
