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
// cand_to_user and user_offsets, groups candidates by user (in the same pass
// for a sorted map, by a stable counting sort otherwise) and derives its own
// work items, so the whole forward is ONE launch.  Larger inputs use the
// separate planning kernel's work list.  When there are more units than
// clusters, items are handed to CTAs in boustrophedon order over the users
// sorted longest first ("Optimizing Jagged Flash Attention with TLX", §2.2:
// tiles sorted by K/V work, even passes left to right, odd passes right to
// left); the items of one (user, head) are adjacent so CTAs sharing a user's
// K/V run together ("In-Kernel Broadcast Optimization", §3.1, Table 1).
//
// K/V are read through tensor maps whose row count is left open, because T
// is only known on the device; the one tile that may reach past row T (the
// tail of the last user) goes through a copy of the map with the row count
// set to T, made by the producer when it first needs it, so the TMA
// zero-fills the missing rows.
//
// Pair mode.  When there are no more (user, head, query tile) units than
// clusters, the two CTAs of a cluster split one unit's keys in half.  Each
// then finishes half of the query rows: it sends O / l and the log-sum-exp
// m + log2(l) of the other half straight into its partner's shared memory
// (asynchronous distributed-shared-memory stores, counted on an mbarrier
// there) and merges what it receives with the log-sum-exp rule of
// "Chapter 4", §4.6.4 (Flash-Decoding): with M = max(m0, lse1),
// out = (2^(m0-M) O0 + 2^(lse1-M) O1/l1) / (2^(m0-M) l0 + 2^(lse1-M)).
//
// Warp roles (384 threads), after the Blackwell design of "Optimizing Jagged
// Flash Attention with TLX", §2.1 (dedicated load, MMA and softmax warps;
// explicit SMEM/TMEM buffers; S/P sharing one TMEM buffer, the PV
// accumulator its own; persistent CTAs):
//   warp 0      TMA producer: Q tile, then K_0, K_1, V_0, K_2, V_1, ... into a
//               ring of shared-memory slots;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T (SS form) into one of two S buffers, then
//               O += P_{j-1} V_{j-1} (TS form, P read from TMEM, one MMA of
//               N = D per 16 keys), so S_j overlaps the softmax of tile j-1;
//   warps 4-11  softmax, O correction and epilogue.  Query row r lives in TMEM
//               lane r; warps 4-7 take key columns 0-63 of every tile and
//               output columns 0..D/2-1, warps 8-11 the other halves, so each
//               row is worked on by two threads that agree on its running
//               maximum through shared memory once per tile.
// Every wait is bounded: a wait that runs out sets the device error word,
// raises an abort flag that ends all roles, and the CTA drains its
// outstanding copies and MMAs before freeing tensor memory.
#pragma once

#include <cuda_bf16.h>

#include <cfloat>

#include "ikbo_common.cuh"
#include "ikbo_ptx.cuh"

namespace ikbo {


constexpr int kBlockN = 128;      // keys per K/V tile
// Each query row is worked on by kSplit threads (column groups of
// kBlockN / kSplit keys), in kSplit x 4 softmax warps after the 4 others.
constexpr int kSplit = 2;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kSoftmaxWarps = 4 * kSplit;
constexpr int kTcThreads = 32 * (kSoftmaxWarp0 + kSoftmaxWarps);
// Hardware barrier 1: warp 0 releases the other warps when the plan is done
// (barrier 0 is __syncthreads).
constexpr int kBarPlanDone = 1;
// The running maximum is moved only when a tile's maximum exceeds it by more
// than this (base-2 units), so un-normalised weights stay <= 2^8 and the
// O correction is skipped on most tiles; the final O / l is exact either way.
constexpr float kLazyRescale = 8.0f;
// Dynamic shared memory: the operand area first (1 KB aligned: 128-byte
// swizzle atoms), the control block after it; 227 KB, the per-CTA maximum.
constexpr int kCtrlBytes = kSplit == 2 ? 3072 : 5120;
constexpr int kDataBytes = 232448 - kCtrlBytes;
constexpr int kTcSmemBytes = kDataBytes + kCtrlBytes;
constexpr int kMaxSlots = 11;
// In-kernel planning keeps off/cand_start/order/prefix (n_user), the per-warp
// counters of the counting sort (kSortWarps x n_user) and cand_to_user/perm
// (n_cand) in the operand area.
constexpr int kFusedMaxUser = 1024;
constexpr int kFusedMaxCand = 20480;
constexpr int kLptMaxUsersFused = 256;
constexpr int kSortWarps = 8;
// Sorted grouping fills cand_start while validating; gaps between
// consecutive users wider than this are filled in a second pass.
constexpr int kSmallGap = 64;

enum TcMode { kModeSkip = -1, kModeListed = 0, kModeIndep = 1, kModePair = 2, kModeClc = 3 };
// SM slots of the Cluster Launch Control tables (indexed by %smid)
constexpr int kClcSlots = 256;
// S/P buffers in tensor memory: the MMA warp computes S two tiles ahead of
// the softmax, so a tile's scores are ready when the softmax gets to it.
constexpr int kSBufs = 3;
constexpr int kCtlItems = 2;

template <int D>
struct TcConfig {
  static constexpr int kCB = D / 64;                   // 128-byte column blocks per row
  static constexpr int kQBytes = kCB * kTileM * 128;    // one Q tile
  static constexpr int kKVBytes = kCB * kBlockN * 128;  // one K or V tile
  // Operand area: two Q buffers, then the K/V ring.  In pair mode only the
  // first Q buffer is used and both together receive the partner's O.
  static constexpr int kFit = (kDataBytes - 2 * kQBytes) / kKVBytes;
  static constexpr int kSlots = kFit < kMaxSlots ? kFit : kMaxSlots;
  static constexpr int kRecvBytes = kTileM * D * 4;
  static constexpr int kPart = D / kSplit;              // output columns per softmax thread
  static constexpr int kOChunk = kPart < 32 ? kPart : 32;   // columns per TMEM load of O
  static constexpr int kOChunks = kPart / kOChunk;
  // tensor-memory columns: three S/P buffers and the O accumulator
  static constexpr int kSCol = 0;
  static constexpr int kOCol = kSBufs * kBlockN;
  static constexpr int kTmemCols = 512;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static_assert(kSlots >= 3, "ring size");
  static_assert(kRecvBytes == 2 * kQBytes, "receive area = both Q buffers");
};

static_assert(kTcSmemBytes <= 232448, "shared memory budget");
static_assert(4 * (4 * (kFusedMaxUser + 1) + kSortWarps * kFusedMaxUser + 2 * kFusedMaxCand) <=
                  kDataBytes,
              "planning scratch");

// Control block, after the operand area.
struct TcCtrl {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots];
  uint64_t s_full[kSBufs], p_full[kSBufs];
  uint64_t pv_done[kSBufs];             // PV of the tile in S buffer i complete
  uint64_t drain, pair_go, pair_recv;
  uint64_t p_half[2];                   // two-tile kernel: first half of P written
  uint32_t tmem_base;
  int abort_flag;
  int mode;
  int n_my_items;
  int sorted;
  int go_sent;
  int total_keys;
  int flags;
  int n_units;                          // planning: units in all (read by every thread)
  int early_loads;                      // ring loads of item 0 issued before the roles start
  union {
    int red[kTcThreads / 32];           // planning: block scan, one word per warp
    int bmaps_ready;                    // after planning: 1 once the bounded V maps are written
  };
  WorkItem items[kCtlItems];            // the first items of this CTA (the rest in global memory)
  union {
    alignas(16) float partner_lse[kTileM];   // one-tile kernel, pair mode
    uint64_t s_free[2];                      // key-interleaved kernel: S buffer read by the softmax
    struct {                                 // two-tile kernel, Cluster Launch Control:
      alignas(16) uint32_t clc_resp[4];      //   the answer to a cancellation request
      uint64_t clc_bar;                      //   ... has arrived
      uint64_t item_full[2];                 //   queue slot k % 2 holds the CTA's k-th item
      uint64_t item_empty[2];                //   every role is done with it
      int lpt;                               //   the tables list the users longest first
    } q;
  };
  int ab_chunk_tiles;                   // key-interleaved kernel: chunk size of split units (0 = none)
  int ab_units;                         // key-interleaved kernel: units (or chunks) in all
  union {
    // row maximum / row sum exchange among the kSplit threads of a row:
    // [parity][column group][row], the value with the exchange's sequence
    // number in its two low bits
    uint32_t xtag[2][kSplit][kTileM];
    // key-interleaved kernel: (running maximum, row sum) of every row, per warpgroup
    float2 ab_ml[2][kTileM];
  };
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
    if (!cluster && ptx::mbar_test_wait(bar, parity)) return true;
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
  // The whole warp waits converged: every lane polls and the warp leaves
  // together, with no divergent branch.  Bounded like wait().
  __device__ __forceinline__ bool conv_wait(uint32_t bar, uint32_t parity) const {
    if (__all_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity))) return true;
    uint64_t t_end = 0;
    for (uint32_t spin = 1;; ++spin) {
      if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
      if (__any_sync(0xffffffffu, *abort != 0)) return false;
      if ((spin & 63u) == 0) {
        const uint64_t now = __shfl_sync(0xffffffffu, ptx::globaltimer(), 0);
        if (t_end == 0) {
          t_end = now + timeout_ns;
        } else if (now > t_end) {
          if ((threadIdx.x & 31) == 0) {
            *abort = 1;
            atomicOr(err_word, kErrTimeout);
          }
          __syncwarp();
          return false;
        }
      }
    }
  }
  // Every lane tests a completed phase at once; otherwise one lane polls and
  // the warp follows its verdict.
  __device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, bool cluster = false) const {
    if (!cluster && __all_sync(0xffffffffu, ptx::mbar_test_wait(bar, parity))) return true;
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

// The same for a kernel whose grid may exceed the buffer's CTAs (the two-tile
// kernel with Cluster Launch Control).  (A separate function: the extra test in
// every call site of trace() cost the one-tile kernel ~1 us of its ~22 us
// launches, which instruction fetch bounds.)
__device__ __forceinline__ void trace_bounded(const AttnParams& p, int ord, int point) {
  if ((int)blockIdx.x < p.trace_ctas) trace(p, ord, point);
}

// Prologue timeline (debug_flags bit 4): item slot 3, points 0..10.
__device__ __forceinline__ void trace_pro(const AttnParams& p, int point) {
  if ((p.debug_flags & 4) && threadIdx.x == 0) trace(p, 3, point);
}

// Per-tile timeline of a CTA's first item (debug_flags bit 2): softmax
// tiles 0-3 in item slot 1 (4 points each), MMA tiles 0-7 in slot 2 (S and
// PV issue).
__device__ __forceinline__ void trace_tile(const AttnParams& p, int k, int slot, int point) {
  if ((p.debug_flags & 2) && k == 0 && point < kTracePoints) trace(p, slot, point);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 32 bf16 values of one output row (16 packed words) to global memory.  A
// warp stores 32 rows at once, each thread its own; with 32-byte stores
// (where the address allows) every thread writes whole 32-byte sectors, two
// instructions instead of four.
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const uint32_t (&w)[16]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
    const size_t a = __cvta_generic_to_global(dst);
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(a), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(a + 32), "r"(w[8]), "r"(w[9]),
                 "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
                 : "memory");
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// A user's last key tile may reach into the rows of the users after it.
// Their keys are masked, so their weights in P are exactly 0, but 0 x inf or
// a NaN in their V rows would spoil P.V ("In-Kernel Broadcast Optimization",
// §3.1: a candidate attends to its own user's sequence only).  So a user's
// last V tile, when it is partial, is loaded through a copy of the V tensor
// map whose row count ends at the user's last row: the TMA fills the rows
// past it with zeros.  The copies live in global memory, one per work item of
// the CTA (slot 2 + k of the CTA's map slots; slots 0 and 1 are the K and V
// maps with the row count T).  One warp without another role writes them all
// right after planning, releases them to the tensor-map proxy with a single
// fence and raises ctl->bmaps_ready; the producer acquires a copy before its
// first load through it.

// Copy `tmpl` into `m` with row count `rows` (one thread; a release fence
// must follow before the TMA may read `m`).
__device__ __forceinline__ void write_bounded_map(CUtensorMap* m, const CUtensorMap* tmpl, int32_t rows) {
  const uint4* s4 = reinterpret_cast<const uint4*>(tmpl);
  uint4* d4 = reinterpret_cast<uint4*>(m);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(d4), "r"(rows) : "memory");
}

// Does item w need a bounded V map (its last tile is partial)?
__device__ __forceinline__ bool needs_bounded_map(const WorkItem& w) { return (w.kv_len % 128) != 0; }

// All threads of one warp: write the bounded V maps of the CTA's n items
// (item_at(k)), release them, set ctl->bmaps_ready.
template <typename ItemAt>
__device__ __forceinline__ void write_bounded_maps(const AttnParams& p, TcCtrl* ctl, const CUtensorMap* vtmpl,
                                                   int n, ItemAt item_at) {
  CUtensorMap* base = p.map_slots + (size_t)p.map_stride * blockIdx.x + 2;
  for (int k = threadIdx.x & 31; k < n; k += 32) {
    const WorkItem w = item_at(k);
    if (needs_bounded_map(w)) write_bounded_map(base + k, vtmpl, w.kv_begin + w.kv_len);
  }
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  __syncwarp();
  if ((threadIdx.x & 31) == 0)
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(ptx::smem_addr(&ctl->bmaps_ready)), "r"(1)
                 : "memory");
}

// All threads of one warp (Cluster Launch Control): a bounded V map for every
// user with candidates whose keys end inside a tile, at maps[user], from the
// CTA's tables (offsets, then first candidates); release them, set
// ctl->bmaps_ready.
__device__ __forceinline__ void write_user_maps(TcCtrl* ctl, CUtensorMap* maps, const CUtensorMap* vtmpl,
                                                const int32_t* off, const int32_t* cs, int n_user) {
  for (int u = threadIdx.x & 31; u < n_user; u += 32)
    if (cs[u + 1] > cs[u] && (off[u + 1] - off[u]) % 128 != 0) write_bounded_map(maps + u, vtmpl, off[u + 1]);
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  __syncwarp();
  if ((threadIdx.x & 31) == 0)
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(ptx::smem_addr(&ctl->bmaps_ready)), "r"(1)
                 : "memory");
}

// The producer's wait for ctl->bmaps_ready (bounded, like every wait).
__device__ __forceinline__ bool wait_bounded_maps(const AttnParams& p, TcCtrl* ctl) {
  uint64_t t_end = 0;
  for (uint32_t spin = 0;; ++spin) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(ptx::smem_addr(&ctl->bmaps_ready))
                 : "memory");
    if (v == 1) return true;
    if ((spin & 63u) == 63u) {
      if (*(volatile int*)&ctl->abort_flag) return false;
      const uint64_t now = ptx::globaltimer();
      if (t_end == 0) {
        t_end = now + p.timeout_ns;
      } else if (now > t_end) {
        ctl->abort_flag = 1;
        atomicOr(p.err_word, kErrTimeout);
        return false;
      }
    }
  }
}

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
    if (lane < nw) red[lane] = w;
  }
  __syncthreads();
  const int pre = warp == 0 ? 0 : red[warp - 1];
  *total = red[nw - 1];
  __syncthreads();
  return pre + v - x;
}

// Inputs (K, V and q together) up to this size are brought into L2 during
// planning: each CTA prefetches its 1/grid share, so that DRAM latency
// overlaps the prologue instead of following it.  Nothing is read twice from
// DRAM for it: the tiles the TMA loads later hit in L2.
constexpr int64_t kPrefetchMaxBytes = int64_t(48) << 20;

// Bulk prefetch instructions are slow to issue, so two threads of different
// warps issue one each, once the offsets are validated: which = 0 for K,
// 2 for q.  Those are what the first MMAs need.
__device__ void prefetch_inputs(const AttnParams& p, int T, int D, int which) {
  const int64_t kv = int64_t(T) * p.H * D * 2;
  const int64_t qb = p.n_cand * p.H * p.Lq * D * 2;
  if (2 * kv + qb > kPrefetchMaxBytes) return;
  const void* base = which == 0 ? (const void*)p.k : (const void*)p.q;
  const int64_t bytes = which == 2 ? qb : kv;
  // byte counts are multiples of 128 (D is 64 or 128), so are the shares
  const int64_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~int64_t(15);
  const int64_t lo = per * blockIdx.x;
  const int64_t hi = lo + per < bytes ? lo + per : bytes;
  if (hi > lo) ptx::prefetch_l2(static_cast<const char*>(base) + lo, uint32_t(hi - lo));
}

// V's share comes after planning, from the two warps (64 threads) that have
// no role once the roles start, one 128-byte line per instruction through
// the load/store path: the DRAM reads of q and K go first, and the TMA unit
// stays free for the first tile loads.  (V prefetched with q and K, or K
// also this way, measured slower: the first tiles' loads waited behind it.)
__device__ __forceinline__ void prefetch_v_late(const AttnParams& p, int T, int D) {
  const int64_t kv = int64_t(T) * p.H * D * 2;
  const int64_t qb = p.n_cand * p.H * p.Lq * D * 2;
  if (2 * kv + qb > kPrefetchMaxBytes) return;
  const int64_t lines = (kv + 127) >> 7;
  const int64_t per = (lines + gridDim.x - 1) / gridDim.x;
  const int64_t lo = per * blockIdx.x;
  const int64_t hi = lo + per < lines ? lo + per : lines;
  for (int64_t l = lo + (threadIdx.x & 63); l < hi; l += 64)
    ptx::prefetch_line_l2(reinterpret_cast<const char*>(p.v) + (l << 7));
}

// ---------------------------------------------------------------------------
// In-kernel planning.  All threads of the CTA; `scratch` is the operand area,
// already holding user_offsets and cand_to_user (plan_load).  Every CTA
// computes the same plan (the inputs are small) and keeps only its own items.
// Few phases, few barriers: on a kernel that runs for microseconds every
// phase costs a barrier and fresh instruction fetches.
// ---------------------------------------------------------------------------
struct PlanScratch {
  int32_t *off, *cs, *order, *ubefore, *wcnt, *c2u, *perm;
  __device__ PlanScratch(uint8_t* base, int n_user, int n_cand) {
    off = reinterpret_cast<int32_t*>(base);   // n_user + 1
    cs = off + (n_user + 1);                  // cand_start, n_user + 1
    order = cs + (n_user + 1);                // n_user
    ubefore = order + n_user;                 // n_user + 1
    wcnt = ubefore + (n_user + 1);            // kSortWarps x n_user (unsorted only)
    c2u = wcnt + kSortWarps * n_user;         // n_cand
    perm = c2u + n_cand;                      // n_cand
  }
};

// kInFlight: loads of each thread in flight at once.  Each round waits for
// its loads (from DRAM when L2 holds no copy), so a large batch of
// candidates wants many: 16384 entries over 384 threads are 11 rounds of 4
// but 3 of 16.  (The one-tile kernel keeps 4: its launches are short and
// bound by instruction fetch, and its batches small.)
template <int kInFlight = 4>
__device__ __forceinline__ void plan_load(const AttnParams& p, uint8_t* scratch) {
  const int n_cand = (int)p.n_cand, n_user = (int)p.n_user;
  PlanScratch S(scratch, n_user, n_cand);
  for (int base = 0; base <= n_user; base += 4 * blockDim.x) {
    int v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = base + i * blockDim.x + threadIdx.x;
      v[i] = u <= n_user ? p.user_offsets[u] : 0;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int u = base + i * blockDim.x + threadIdx.x;
      if (u <= n_user) S.off[u] = v[i];
    }
  }
  for (int base = 0; base < n_cand; base += kInFlight * blockDim.x) {
    int v[kInFlight];
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      const int c = base + i * blockDim.x + threadIdx.x;
      v[i] = c < n_cand ? p.cand_to_user[c] : 0;
    }
    if (p.vendor_to_user) {
      // a multi-level call: the loaded values are vendors; an out-of-range
      // one becomes -1, which the validation reports as a bad index
#pragma unroll
      for (int i = 0; i < kInFlight; ++i)
        v[i] = (v[i] >= 0 && int64_t(v[i]) < p.n_vendor) ? p.vendor_to_user[v[i]] : -1;
    }
#pragma unroll
    for (int i = 0; i < kInFlight; ++i) {
      const int c = base + i * blockDim.x + threadIdx.x;
      if (c < n_cand) S.c2u[c] = v[i];
    }
  }
}

// Flags found while validating and grouping.
constexpr int kPlanBadOff = 1, kPlanBadIdx = 2, kPlanUnsorted = 4, kPlanEmpty = 8, kPlanGap = 16;

// Validation and grouping, all threads of the CTA (the first part of every
// in-kernel plan).  On return cand_start (the scratch's `cs`) holds the first
// grouped position of every user, `perm_ws` the grouped order when the map
// is unsorted, and the rows of candidates whose user has an empty sequence
// are zero.  Returns the flags, or -1 when the index tensors are invalid:
// then the CTA has no work (mode kModeSkip) and CTA 0 has set the error word.
__device__ int plan_group(const AttnParams& p, TcCtrl* ctl, uint8_t* scratch, int D,
                          bool prefetch = true) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int grid = gridDim.x, b = blockIdx.x;
  const int n_cand = (int)p.n_cand, n_user = (int)p.n_user;
  PlanScratch S(scratch, n_user, n_cand);
  int32_t* const off = S.off;
  int32_t* const cs = S.cs;
  int32_t* const c2u = S.c2u;
  constexpr int kBadOff = kPlanBadOff, kBadIdx = kPlanBadIdx, kUnsorted = kPlanUnsorted,
                kEmpty = kPlanEmpty, kGap = kPlanGap;

  // One pass: validation, sortedness, empty sequences, and for sorted input
  // the first candidate of every user (users prev+1 .. x start at c).
  int flags = 0;
  if (tid == 0 && off[0] != 0) flags |= kBadOff;
  // a fused self-attention call states T: the offsets must end there
  if (tid == 0 && p.q_user && (int64_t)off[n_user] != p.total_rows) flags |= kBadOff;
  for (int u = tid; u < n_user; u += nt) {
    if (off[u + 1] < off[u]) flags |= kBadOff;
    if (off[u + 1] == off[u]) flags |= kEmpty;
  }
  for (int c = tid; c < n_cand; c += nt) {
    const int x = c2u[c];
    const int prev = c == 0 ? -1 : c2u[c - 1];
    if (x < 0 || x >= n_user) flags |= kBadIdx;
    if (prev > x) {
      flags |= kUnsorted;
    } else if (prev < x && x < n_user) {
      if (x - prev <= kSmallGap) {
        for (int uu = max(prev + 1, 0); uu <= x; ++uu) cs[uu] = c;
      } else {
        flags |= kGap;
      }
    }
    if (c == n_cand - 1 && x >= 0 && x < n_user) {
      if (n_user - x <= kSmallGap) {
        for (int uu = x + 1; uu <= n_user; ++uu) cs[uu] = n_cand;
      } else {
        flags |= kGap;
      }
    }
  }
  // no candidates at all (a self-attention-only call): the pass above wrote
  // no cand_start entry, and every user has zero candidates
  if (n_cand == 0)
    for (int u = tid; u <= n_user; u += nt) cs[u] = 0;
  if (flags) atomicOr(&ctl->flags, flags);
  __syncthreads();
  flags = ctl->flags;
  trace_pro(p, 4);
  if (flags & (kBadOff | kBadIdx)) {
    if (tid == 0) {
      ctl->mode = kModeSkip;
      ctl->n_my_items = 0;
      ctl->sorted = 1;
      if (b == 0)
        atomicOr(p.err_word, ((flags & kBadOff) ? kErrOffsets : 0) | ((flags & kBadIdx) ? kErrIndex : 0));
    }
    __syncthreads();
    return -1;
  }
  // the offsets are valid: start the DRAM reads of this CTA's share of the
  // inputs (lane 0 of warps 1-3)
  if (prefetch && (tid == 32 || tid == 96)) prefetch_inputs(p, off[n_user], D, (tid >> 5) - 1);
  const bool unsorted = (flags & kUnsorted) != 0;
  if (!unsorted && (flags & kGap)) {
    // sorted, with wide gaps between consecutive users: fill those now
    for (int c = tid; c < n_cand; c += nt) {
      const int x = c2u[c];
      const int prev = c == 0 ? -1 : c2u[c - 1];
      if (x - prev > kSmallGap)
        for (int uu = prev + 1; uu <= x; ++uu) cs[uu] = c;
      if (c == n_cand - 1 && n_user - x > kSmallGap)
        for (int uu = x + 1; uu <= n_user; ++uu) cs[uu] = n_cand;
    }
    __syncthreads();
  }
  if (unsorted) {
    // stable counting sort: sort warp w < kSortWarps owns a contiguous segment
    // of candidates; the other warps only take part in the barriers
    int32_t* const wcnt = S.wcnt;
    int32_t* const perm = S.perm;
    const int warp = tid >> 5, lane = tid & 31, nw = kSortWarps;
    const bool sorter = warp < nw;
    const int seg = (n_cand + nw - 1) / nw;
    const int seg_end = sorter ? min(n_cand, (warp + 1) * seg) : 0;
    for (int i = tid; i < nw * n_user; i += nt) wcnt[i] = 0;
    __syncthreads();
    if (sorter)
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
      const int ex = block_scan_excl(tot_u, ctl->red, &tot);
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
    for (int base = warp * seg; sorter && base < seg_end; base += 32) {
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
  trace_pro(p, 5);
  // rows of candidates whose user has an empty sequence are zero
  if (flags & kEmpty) {
    const int64_t elems = (int64_t)p.H * p.Lq * D;
    for (int c = b * nt + tid; c < n_cand; c += grid * nt) {
      const int x = c2u[c];
      if (off[x + 1] == off[x]) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)c * elems);
        for (int64_t i = 0; i < elems / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  return flags;
}

// A unit is (user, head, up to tiles_per_unit query tiles of the user's
// candidates): 1 for this kernel, 2 for the two-tile kernel.
// Unit i of the plan as a work item: user rank lo, the last with
// ubefore[lo] <= i (users by rank: order, or index order when null), then its
// head and query tile.  The tables are the planning scratch in shared memory,
// or a CTA's copy in global memory (Cluster Launch Control).
__device__ __forceinline__ void decode_unit(int i, const int32_t* off, const int32_t* cs,
                                            const int32_t* ubefore, const int32_t* order, int n_user,
                                            int tiles_per_unit, int cands_per_tile, bool self_tiles,
                                            WorkItem& w) {
  const int cpt = cands_per_tile * tiles_per_unit;   // candidates per unit
  const int srows = kTileM * tiles_per_unit;         // sequence rows per self-attention unit
  int lo = 0, hi = n_user - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ubefore[mid] <= i) lo = mid; else hi = mid - 1;
  }
  const int u = order ? order[lo] : lo;
  const int r = cs[u + 1] - cs[u];
  const int L = off[u + 1] - off[u];
  const int nmt = r > 0 ? ceil_div(r, cpt) : 0;
  const int per_head = nmt + (self_tiles ? ceil_div(L, srows) : 0);
  const int local = i - ubefore[lo];
  const int h = local / per_head, mt = local - h * per_head;
  w.user = u;
  w.head = h;
  if (mt < nmt) {
    w.cand_begin = cs[u] + mt * cpt;
    w.n_cand = min(cpt, r - mt * cpt);
    w.q_row = -1;
  } else {
    // tiles of the user's own sequence (self-attention): up to srows rows
    const int t = mt - nmt;
    w.cand_begin = 0;
    w.n_cand = min(srows, L - t * srows);
    w.q_row = off[u] + t * srows;
  }
  w.kv_begin = off[u];
  w.kv_len = L;
  w.unit = -1;
  w.unit_first = 0;
  // two-tile kernel: a user's only query tile may have its keys split over
  // the two warpgroups
  w.n_split = (tiles_per_unit == 2 && mt < nmt && r <= cands_per_tile) ? 2 : 1;
}

// kClc (two-tile kernel with Cluster Launch Control, clc_tables non-null):
// the units are not dealt; the plan's user tables go to this global slot
// instead, from which the CTA decodes unit blockIdx.x and those of the CTAs it
// takes over.  (A template parameter, so that the one-tile kernel, whose
// short launches are bound by instruction fetch, carries none of that code.)
template <bool kClc = false>
__device__ void plan_in_cta(const AttnParams& p, TcCtrl* ctl, uint8_t* scratch, int D,
                            int tiles_per_unit, int32_t* clc_tables = nullptr) {
  const int flags = plan_group(p, ctl, scratch, D);
  if (flags < 0) return;
  const bool unsorted = (flags & kPlanUnsorted) != 0;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int grid = gridDim.x, b = blockIdx.x;
  const int n_cand = (int)p.n_cand, n_user = (int)p.n_user;
  PlanScratch S(scratch, n_user, n_cand);
  int32_t* const off = S.off;
  int32_t* const cs = S.cs;
  int32_t* const order = S.order;
  int32_t* const ubefore = S.ubefore;
  (void)n_cand;
  // Units (H x groups of query tiles of users with candidates and keys),
  // prefix-summed over the users in index order, or longest first (below).
  const int cpt = p.cands_per_tile * tiles_per_unit;   // candidates per unit
  const int srows = kTileM * tiles_per_unit;           // sequence rows per self-attention unit
  bool lpt = false;
  auto user_at = [&](int rk) { return lpt ? order[rk] : rk; };
  auto units_of = [&](int u) {
    const int r = cs[u + 1] - cs[u], L = off[u + 1] - off[u];
    if (L <= 0) return 0;
    // candidate tiles, plus (fused self-attention) the user's own sequence
    // in units of tiles_per_unit tiles of 128 rows
    const int tiles = (r > 0 ? ceil_div(r, cpt) : 0) + (p.q_user ? ceil_div(L, srows) : 0);
    return p.H * tiles;
  };
  auto prefix = [&]() {
    if (n_user <= 32) {
      if (tid < 32) {
        const int nu = tid < n_user ? units_of(user_at(tid)) : 0;
        int v = nu;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, v, o);
          if (tid >= o) v += y;
        }
        if (tid < n_user) ubefore[tid] = v - nu;
        if (tid == 31) {
          ubefore[n_user] = v;
          ctl->n_units = v;
        }
      }
    } else {
      int carry = 0;
      for (int base = 0; base < n_user; base += nt) {
        const int rk = base + tid;
        const int nu = rk < n_user ? units_of(user_at(rk)) : 0;
        int tot;
        const int ex = block_scan_excl(nu, ctl->red, &tot);
        if (rk < n_user) ubefore[rk] = carry + ex;
        carry += tot;
      }
      if (tid == 0) {
        ubefore[n_user] = carry;
        ctl->n_units = carry;
      }
    }
    // the scratch may be overwritten by TMA (async proxy) once the decode
    // that follows is done
    ptx::fence_proxy_async_smem();
    __syncthreads();
  };
  prefix();
  // from the control block: after this barrier only thread 0 reads the
  // scratch (the pair-mode decode), so it may start the TMA into it
  const int N = ctl->n_units;
  // Pair mode when every unit gets a cluster of its own; otherwise units are
  // dealt to independent CTAs, users longest first.
  const bool pair = tiles_per_unit == 1 && N > 0 && 2 * N <= grid;
  if (!pair && n_user > 1 && n_user <= kLptMaxUsersFused) {
    __syncthreads();   // everyone has read N before the prefix is rewritten
    for (int u = tid; u < n_user; u += nt) {
      const int Lu = off[u + 1] - off[u];
      int rank = 0;
      for (int w = 0; w < n_user; ++w) {
        const int Lw = off[w + 1] - off[w];
        rank += (Lw > Lu) || (Lw == Lu && w < u);
      }
      order[rank] = u;
    }
    lpt = true;
    __syncthreads();
    prefix();
  }
  trace_pro(p, 6);
  if (kClc && clc_tables) {
    const int n1 = n_user + 1;
    for (int j = tid; j < n1; j += nt) {
      clc_tables[j] = off[j];
      clc_tables[n1 + j] = cs[j];
      clc_tables[2 * n1 + j] = ubefore[j];
      clc_tables[3 * n1 + j] = (lpt && j < n_user) ? order[j] : j;
    }
    if (tid == 0) {
      ctl->mode = kModeClc;
      ctl->sorted = unsorted ? 0 : 1;
      ctl->total_keys = off[n_user];
      ctl->n_my_items = 0;
      ctl->q.lpt = lpt ? 1 : 0;
    }
    return;
  }
  // decode unit i into a work item
  auto decode = [&](int i, WorkItem& w) {
    decode_unit(i, off, cs, ubefore, lpt ? order : nullptr, n_user, tiles_per_unit, p.cands_per_tile,
                p.q_user != nullptr, w);
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
          ctl->items[0] = w;
          count = 1;
        } else if (rank == 0) {
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
      if (k < kCtlItems) ctl->items[k] = w; else mine[k] = w;
    }
    if (tid == 0) ctl->n_my_items = count;
  }
  if (tid == 0) {
    ctl->mode = pair ? kModePair : kModeIndep;
    ctl->sorted = unsorted ? 0 : 1;
    ctl->total_keys = off[n_user];
  }
  // no closing barrier: the kernel's follows (after thread 0 may have
  // started the first TMA loads)
}

// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
ikbo_attn_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap qmap1,
                    const __grid_constant__ CUtensorMap kmap_tmpl,
                    const __grid_constant__ CUtensorMap vmap_tmpl,
                    const __grid_constant__ CUtensorMap qumap) {
  using C = TcConfig<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* data = smem_raw;
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem_raw + kDataBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t cta_rank = ptx::cluster_ctarank();
  // 128-byte swizzle atoms must start on 1 KB boundaries
  const bool layout_ok = (ptx::smem_addr(smem_raw) & 1023u) == 0;
  trace_pro(p, 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->q_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->q_empty[i]), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[i]), kSoftmaxWarps);
      ptx::mbar_init(ptx::smem_addr(&ctl->pv_done[i]), 1);
    }
    for (int i = 0; i < kMaxSlots; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_go), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_recv), 1);
    ctl->go_sent = 0;
    ctl->abort_flag = 0;
    ctl->flags = 0;
    ctl->early_loads = -1;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // exchange words start with sequence number 3, which no first use expects
  for (int i = threadIdx.x; i < 2 * kSplit * kTileM; i += blockDim.x) (&ctl->xtag[0][0][0])[i] = 3u;
  if (warp == 2 && lane == 0) {
    // the host-encoded descriptors into the TMA unit's cache ahead of use
    if (p.n_cand > 0) ptx::prefetch_tensormap(&qmap);   // a self-only call encodes no Q map
    ptx::prefetch_tensormap(&kmap_tmpl);
    ptx::prefetch_tensormap(&vmap_tmpl);
    if (p.q_user) ptx::prefetch_tensormap(&qumap);
  }
  // A planning kernel may precede this one (programmatic dependent launch):
  // its work list is visible after this wait.  Without one it returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (p.fused && layout_ok) plan_load(p, data);
  __syncthreads();
  // Split cluster barrier (every thread, warps converged): arrive now, this
  // CTA's barriers being initialised; wait once planning is done, before any
  // access to the partner's shared memory.  The partner has long arrived by
  // then, so the wait costs nothing.
  ptx::cluster_arrive_relaxed();
  trace_pro(p, 1);
  if (!layout_ok) {
    if (threadIdx.x == 0) {
      ctl->mode = kModeSkip;
      ctl->n_my_items = 0;
      ctl->sorted = 1;
      atomicOr(p.err_word, kErrLayout);
    }
  } else if (p.fused) {
    plan_in_cta(p, ctl, data, D, 1);
    trace_pro(p, 7);
    // the planning scratch is overwritten by TMA (async proxy) from here on
    ptx::fence_proxy_async_smem();
  } else if (threadIdx.x == 0) {
    ctl->mode = kModeListed;
    ctl->sorted = p.header->sorted != 0;
    ctl->total_keys = p.header->total_keys;
    const int n = p.header->n_items;
    ctl->n_my_items =
        n > (int)blockIdx.x ? (n - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  }

  uint8_t* q_smem = data;
  uint8_t* kv_smem = data + 2 * C::kQBytes;
  const int32_t* perm = p.fused ? p.perm_ws : p.perm;
  const int Lq = p.Lq;
  // ---- TMA issue, used by the producer (and by thread 0, the producer's
  // lane, to start a pair item's loads before the other roles start)
  bool tail_ready = false;
  // Fused mode loads through the host maps, whose row count is open; a tile
  // that reaches past row T goes through a copy with the row count set to T
  // (made on first need), so the TMA fills its missing rows with zeros
  // instead of reading past the end of k / v.
  auto kv_map = [&](bool is_v, int32_t row) -> const void* {
    if (!p.fused) return is_v ? p.vmap : p.kmap;
    // maps encoded with the row count T itself (the caller stated T)
    if (p.exact_rows) return is_v ? (const void*)&vmap_tmpl : (const void*)&kmap_tmpl;
    const int T = ctl->total_keys;
    if (row + kBlockN <= T) return is_v ? (const void*)&vmap_tmpl : (const void*)&kmap_tmpl;
    CUtensorMap* tail_k = p.map_slots + (size_t)p.map_stride * blockIdx.x;
    CUtensorMap* tail_v = tail_k + 1;
    if (!tail_ready) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const uint4* s4 = reinterpret_cast<const uint4*>(mi == 0 ? &kmap_tmpl : &vmap_tmpl);
        uint4* d4 = reinterpret_cast<uint4*>(mi == 0 ? tail_k : tail_v);
#pragma unroll
        for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
        asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(d4), "r"(T)
                     : "memory");
      }
      asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
      ptx::tensormap_acquire(tail_k);
      ptx::tensormap_acquire(tail_v);
      tail_ready = true;
    }
    return is_v ? (const void*)tail_v : (const void*)tail_k;
  };
  // The V map for the tile at `row` of the CTA's item k, whose keys end at
  // row `end`: a user's partial last tile goes through the item's bounded
  // copy (the TMA fills the other users' rows with zeros).
  bool bm_ready = false;
  auto v_map_for = [&](int32_t row, int32_t end, int k) -> const void* {
    if (row + kBlockN <= end) return kv_map(true, row);
    if (!bm_ready) {
      if (!wait_bounded_maps(p, ctl)) return nullptr;
      bm_ready = true;
    }
    CUtensorMap* m = p.map_slots + (size_t)p.map_stride * blockIdx.x + 2 + k;
    ptx::tensormap_acquire(m);
    ptx::prefetch_tensormap(m);
    return m;
  };
  // the map of a K or V tile at `row` of the CTA's item k, whose keys end at
  // row `end` (null after an abort)
  auto map_for = [&](bool is_v, int32_t row, int32_t end, int k) -> const void* {
    return is_v ? v_map_for(row, end, k) : kv_map(false, row);
  };
  // one K or V tile (128 keys x D of one head) into ring slot `slot` through `map`
  auto issue_tile = [&](const void* map, int head, int32_t row, uint32_t slot) -> bool {
    if (!map) return false;
    const uint32_t bar = ptx::smem_addr(&ctl->kv_full[slot]);
    const uint32_t dst = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
    ptx::mbar_arrive_expect_tx(bar, C::kKVBytes);
#pragma unroll
    for (int cb = 0; cb < C::kCB; ++cb)
      ptx::tma_load_2d(dst + cb * kBlockN * 128, map, bar, head * D + cb * 64, row);
    return true;
  };
  // the Q tile of item w into Q buffer qb
  auto issue_q = [&](const WorkItem& w, uint32_t qb) {
    const uint32_t qbar = ptx::smem_addr(&ctl->q_full[qb]);
    const uint32_t qdst = ptx::smem_addr(q_smem + qb * C::kQBytes);
    if (w.q_row >= 0) {
      // 128 rows of the user sequence's queries (rows past T read as zeros)
      ptx::mbar_arrive_expect_tx(qbar, uint32_t(C::kCB * kTileM * 128));
#pragma unroll
      for (int cb = 0; cb < C::kCB; ++cb)
        ptx::tma_load_2d(qdst + cb * kTileM * 128, &qumap, qbar, w.head * D + cb * 64, w.q_row);
    } else if (ctl->sorted) {
      const int nb = p.qbox;
      const int nbox = ceil_div(w.n_cand, nb);
      ptx::mbar_arrive_expect_tx(qbar, uint32_t(nbox * nb * Lq * 128 * C::kCB));
      for (int cb = 0; cb < C::kCB; ++cb)
        for (int bx = 0; bx < nbox; ++bx)
          ptx::tma_load_4d(qdst + cb * kTileM * 128 + bx * nb * Lq * 128, &qmap, qbar, cb * 64, 0, w.head,
                           w.cand_begin + bx * nb);
    } else {
      ptx::mbar_arrive_expect_tx(qbar, uint32_t(w.n_cand * Lq * 128 * C::kCB));
      for (int i = 0; i < w.n_cand; ++i) {
        const int32_t c = perm[w.cand_begin + i];
        for (int cb = 0; cb < C::kCB; ++cb)
          ptx::tma_load_4d(qdst + cb * kTileM * 128 + i * Lq * 128, &qmap1, qbar, cb * 64, 0, w.head, c);
      }
    }
  };
  // The i-th ring load of an item of n tiles, in the MMA warp's order
  // K0, K1, K2, V0, K3, V1, K4, ..., V(n-1): is it V, and which tile.
  auto load_at = [](int i, int n, bool& is_v, int& tile) {
    const int k0 = n < kSBufs ? n : kSBufs;
    const int a = n > kSBufs ? n - kSBufs : 0;   // tiles j followed by K(j+3)
    if (i < k0) {
      is_v = false;
      tile = i;
    } else if (i - k0 < 2 * a) {
      const int t = i - k0;
      is_v = (t & 1) == 0;
      tile = is_v ? (t >> 1) : (t >> 1) + kSBufs;
    } else {
      is_v = true;
      tile = a + (i - k0 - 2 * a);
    }
  };
  if (threadIdx.x == 0) {
    trace(p, 0, kTrCtaStart);
    ctl->bmaps_ready = 0;   // the planning's scan words are free now
  }
  ptx::tc_fence_before();
  if (warp == 0) {
    // The plan is complete: warp 0 releases the other warps and only then
    // starts a pair item's loads.  One warp arrives while the others wait,
    // so this takes the non-aligned barrier forms on a barrier of its own
    // (the aligned ones require every thread to run the same instruction).
    asm volatile("barrier.arrive %0, %1;" ::"r"(kBarPlanDone), "r"(kTcThreads) : "memory");
    if (lane == 0 && p.fused && ctl->mode == kModePair && ctl->n_my_items > 0 && !(p.debug_flags & 1)) {
      // Pair item: start its Q and the first ring loads now, while the other
      // warps set out.  Since the last planning barrier only this thread has
      // read the scratch that the loads overwrite.
      ptx::fence_proxy_async_smem();
      const WorkItem w = ctl->items[0];
      const int n = ceil_div(w.kv_len, kBlockN);
      issue_q(w, 0);
      int e = 0;
      for (; e < 2 * n && e < C::kSlots; ++e) {
        bool is_v;
        int t;
        load_at(e, n, is_v, t);
        const int32_t row = w.kv_begin + t * kBlockN;
        if (!issue_tile(map_for(is_v, row, w.kv_begin + w.kv_len, 0), w.head, row, (uint32_t)e)) break;
      }
      ctl->early_loads = e;
    }
    __syncwarp();
  } else {
    asm volatile("barrier.sync %0, %1;" ::"r"(kBarPlanDone), "r"(kTcThreads) : "memory");
  }
  ptx::cluster_wait();
  ptx::tc_fence_after();
  trace_pro(p, 8);

  const uint32_t tmem = ctl->tmem_base;
  const int mode = ctl->mode;
  const int n_my = ctl->n_my_items;
  const bool sorted = ctl->sorted != 0;
  const int NS = C::kSlots;
  const int NQ = mode == kModePair ? 1 : 2;
  const Waiter W{&ctl->abort_flag, p.err_word, p.timeout_ns};
  auto item_at = [&](int k) -> WorkItem {
    if (p.fused) return k < kCtlItems ? ctl->items[k] : p.cta_items[(size_t)blockIdx.x * p.max_cta_items + k];
    return p.items[blockIdx.x + (size_t)k * gridDim.x];
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && mode != kModeSkip) {
      if (!p.fused) {
        ptx::tensormap_acquire(p.kmap);
        ptx::tensormap_acquire(p.vmap);
      }
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      for (int k = 0; k < n_my && ok; ++k) {
        const WorkItem w = item_at(k);
        const int n = ceil_div(w.kv_len, kBlockN);
        // item 0 of a pair may have been started before the roles began
        const int e0 = (k == 0 && ctl->early_loads >= 0) ? ctl->early_loads : 0;
        const uint32_t qb = q_it % NQ;
        trace(p, k, kTrProdItem);
        if (!(k == 0 && ctl->early_loads >= 0)) {
          if (!W.wait(ptx::smem_addr(&ctl->q_empty[qb]), ((q_it / NQ) & 1u) ^ 1u)) break;
          if (!(p.debug_flags & 1)) issue_q(w, qb);
        }
        ++q_it;
        kv_it += (uint32_t)e0;
        for (int i = e0; i < 2 * n; ++i) {
          bool is_v;
          int t;
          load_at(i, n, is_v, t);
          const uint32_t slot = kv_it % NS;
          // the map first: a bounded map's acquire and descriptor fetch then
          // overlap the wait for the slot
          const int32_t row = w.kv_begin + t * kBlockN;
          const void* map = map_for(is_v, row, w.kv_begin + w.kv_len, k);
          if (!map || !W.wait(ptx::smem_addr(&ctl->kv_empty[slot]), ((kv_it / NS) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          if (!issue_tile(map, w.head, row, slot)) {
            ok = false;
            break;
          }
          ++kv_it;
        }
        trace(p, k, kTrProdIssued);
        if (ok && w.unit >= 0) {
          // pair item: once the last S has read Q, the Q buffers can receive
          // the partner's O / l and log-sum-exp of the rows this CTA finishes
          // (the first half for CTA 0, the second for CTA 1); tell the partner
          if (!W.wait(ptx::smem_addr(&ctl->q_empty[0]), 0)) break;
          const int rows = w.q_row >= 0 ? w.n_cand : w.n_cand * Lq, hrows = (rows + 1) >> 1;
          const int recv = cta_rank == 0 ? hrows : rows - hrows;
          ptx::mbar_arrive_expect_tx(ptx::smem_addr(&ctl->pair_recv), uint32_t(recv * (D * 4 + 4)));
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
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kTileM, D, 1);
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
        // S_j = Q K_j^T into S buffer (g + j) % 3
        auto issue_s = [&](int j) -> bool {
          const uint32_t slot = kv_it % NS;
          if (!W.wait(ptx::smem_addr(&ctl->kv_full[slot]), (kv_it / NS) & 1u)) return false;
          ptx::tc_fence_after();
          const uint32_t k_base = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
          const uint32_t sb = (g + j) % kSBufs;
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
          if (j < 8) trace_tile(p, k, 2, 2 * j);
          ptx::mma_commit(ptx::smem_addr(&ctl->kv_empty[slot]));
          ptx::mma_commit(ptx::smem_addr(&ctl->s_full[sb]));
          if (j == n - 1) ptx::mma_commit(ptx::smem_addr(&ctl->q_empty[qb]));
          ++kv_it;
          return true;
        };
        for (int j = 0; j < n && j < kSBufs && ok; ++j) ok = issue_s(j);
        for (int j = 0; j < n && ok; ++j) {
          // O += P_j V_j once the softmax has written P_j over S_j
          const uint32_t gj = g + j;
          const uint32_t pb = gj % kSBufs;
          if (!W.wait(ptx::smem_addr(&ctl->p_full[pb]), (gj / kSBufs) & 1u)) {
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
          // V is MN-major (d contiguous): 8-key groups 1 KB apart, the two
          // 64-column blocks of a D = 128 tile kBlockN * 128 bytes apart
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            const uint64_t bdesc = ptx::smem_desc_sw128(v_base + kk * 16 * 128, kBlockN * 128, 1024);
            ptx::mma_ts(tmem + C::kOCol, a_tmem + kk * 8, bdesc, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          }
          if (j < 8) trace_tile(p, k, 2, 2 * j + 1);
          ptx::mma_commit(ptx::smem_addr(&ctl->kv_empty[slot]));
          ptx::mma_commit(ptx::smem_addr(&ctl->pv_done[pb]));
          if (j == n - 1) trace(p, k, kTrMmaLastPV);
          ++kv_it;
          // the S buffer of P_j is free once PV_j has read it (MMAs run in order)
          if (j + kSBufs < n) ok = issue_s(j + kSBufs);
        }
        g += n;
        ++q_it;
      }
      // All issued MMAs must finish before tensor memory is released.
      ptx::mma_commit(ptx::smem_addr(&ctl->drain));
      W.drain(ptx::smem_addr(&ctl->drain), 0);
    }
    __syncwarp();
  } else if (warp == 2) {
    if (mode != kModeSkip)
      write_bounded_maps(p, ctl, p.fused ? &vmap_tmpl : static_cast<const CUtensorMap*>(p.vmap), n_my, item_at);
  } else if (warp >= kSoftmaxWarp0 && mode != kModeSkip) {
    // ------------------------------------------- softmax / correction / epilogue
    constexpr int kCols = kBlockN / kSplit;                  // key columns of a tile per thread
    constexpr int kR = kCols / 32;                           // 32-column TMEM loads per tile
    const int quarter = warp & 3;
    const int cg = (warp - kSoftmaxWarp0) >> 2;              // column group of this thread
    const int row = quarter * 32 + lane;                     // TMEM lane == tile row
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, xs = 0;
    // PV(x) commits to pv_done[x % 3], phase x / 3.  A wait for PV(x) is
    // made only on tile x + 1 (to rescale O) or after the item's last tile
    // x: by then S(x) is complete, so PV(x - 3), the barrier's previous
    // phase, is complete (the MMA warp issues S(x) after it), and PV(x + 3),
    // its next phase, needs this warp's p_full(x + 3).  The parity of the
    // phase is therefore unambiguous without observing every phase.
    // PV(x) complete implies every earlier PV complete (MMAs run in order).
    auto pv_wait = [&](uint32_t x) -> bool {
      if (!W.warp_wait(ptx::smem_addr(&ctl->pv_done[x % kSBufs]), (x / kSBufs) & 1u)) return false;
      ptx::tc_fence_after();
      return true;
    };
    // Row values shared among the kSplit threads of a row: a value goes out
    // with the exchange's sequence number in its two low bits (it moves by at
    // most 3 ulp; -inf and NaN go out as -FLT_MAX), and a partner's word is
    // taken once it carries the same number.  Every thread of the row then
    // holds the same kSplit words.  The waits are bounded like every wait.
    auto publish = [&](float v) -> uint32_t {
      const float vv = v > -FLT_MAX ? v : -FLT_MAX;
      const uint32_t wv = (__float_as_uint(vv) & ~3u) | (xs & 3u);
      asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(
                       ptx::smem_addr(&ctl->xtag[xs & 1u][cg][row])),
                   "r"(wv)
                   : "memory");
      return wv;
    };
    auto collect = [&](uint32_t mine, uint32_t (&words)[kSplit]) -> bool {
      const uint32_t tag = xs & 3u, par = xs & 1u;
      ++xs;
      bool ok = true;
      uint64_t t_end = 0;
#pragma unroll
      for (int o = 0; o < kSplit; ++o) {
        if (o == cg) {
          words[o] = mine;
          continue;
        }
        const uint32_t addr = ptx::smem_addr(&ctl->xtag[par][o][row]);
        uint32_t wv = 0;
        for (uint32_t spin = 0; ok; ++spin) {
          asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(wv) : "r"(addr) : "memory");
          if ((wv & 3u) == tag) break;
          if ((spin & 127u) == 127u) {
            if (*W.abort) {
              ok = false;
              break;
            }
            const uint64_t now = ptx::globaltimer();
            if (t_end == 0) {
              t_end = now + p.timeout_ns;
            } else if (now > t_end) {
              *W.abort = 1;
              atomicOr(p.err_word, kErrTimeout);
              ok = false;
            }
          }
        }
        words[o] = wv;
      }
      return __all_sync(0xffffffffu, ok);
    };
    auto dec = [](uint32_t wv) { return __uint_as_float(wv & ~3u); };
    for (int k = 0; k < n_my; ++k) {
      const WorkItem w = item_at(k);
      const int n = ceil_div(w.kv_len, kBlockN);
      const int rows = w.q_row >= 0 ? w.n_cand : w.n_cand * Lq;   // query rows of the tile
      // Rows past the item's queries hold stale shared memory; their results
      // are never stored, and they are left out of every decision below.
      const bool live = row < rows;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj % kSBufs;
        if (!W.warp_wait(ptx::smem_addr(&ctl->s_full[sb]), (gj / kSBufs) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (j == 0 && row == 0 && cg == 0) trace(p, k, kTrSmS0);
        const bool tr_t = row == 0 && cg == 0 && j < 4;
        if (tr_t) trace_tile(p, k, 1, 4 * j);
        const uint32_t scol = tmem + lane_off + C::kSCol + sb * kBlockN;
        uint32_t r[kR][32];
#pragma unroll
        for (int c = 0; c < kR; ++c) ptx::tmem_ld32(scol + cg * kCols + c * 32, r[c]);
        ptx::tmem_ld_wait();
#define IKBO_S(e) __uint_as_float(r[(e) >> 5][(e) & 31])
        // Scores enter the exponent as fma(s, sc, -ref).  On a tile whose
        // tail is short, or for scale <= 0, they are scaled here first and
        // the missing keys set to -inf (sc = 1); otherwise sc = scale and the
        // order of the raw scores is that of the scaled ones.
        const int valid = min(kBlockN, w.kv_len - j * kBlockN) - cg * kCols;
        float sc = sl2;
        if (valid < kCols || !(sl2 > 0.f)) {
#pragma unroll
          for (int e = 0; e < kCols; ++e) {
            const float tt = IKBO_S(e) * sl2;
            r[e >> 5][e & 31] = __float_as_uint(e < valid ? tt : -INFINITY);
          }
          sc = 1.f;
        }
        float mx;
        {
          // four independent chains
          float a0 = fmaxf(IKBO_S(0), IKBO_S(1)), a1 = fmaxf(IKBO_S(2), IKBO_S(3));
          float a2 = fmaxf(IKBO_S(4), IKBO_S(5)), a3 = fmaxf(IKBO_S(6), IKBO_S(7));
#pragma unroll
          for (int e = 8; e < kCols; e += 8) {
            a0 = fmax3(a0, IKBO_S(e), IKBO_S(e + 1));
            a1 = fmax3(a1, IKBO_S(e + 2), IKBO_S(e + 3));
            a2 = fmax3(a2, IKBO_S(e + 4), IKBO_S(e + 5));
            a3 = fmax3(a3, IKBO_S(e + 6), IKBO_S(e + 7));
          }
          mx = fmax3(a0, a1, fmaxf(a2, a3)) * sc;
        }
        // This thread's S reads are complete: the others of the row may write
        // P over them once they have seen this maximum.
        ptx::tc_fence_before();
        if (tr_t) trace_tile(p, k, 1, 4 * j + 1);
        const uint32_t mx_w = publish(mx);
        // P = 2^(t - ref) as bf16 pairs, and its row sum
        uint32_t pk[kCols / 2];
        float sum = 0.f;
        auto exps = [&](float ref) {
          const float2 sc2 = make_float2(sc, sc), nr2 = make_float2(-ref, -ref);
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < kCols; e += 2) {
            const float2 x = ffma2(make_float2(IKBO_S(e), IKBO_S(e + 1)), sc2, nr2);
            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            if ((e >> 1) & 1) a1 = fadd2(a1, pe); else a0 = fadd2(a0, pe);
            pk[e >> 1] = pack_bf16(pe.x, pe.y);
          }
          const float2 u = fadd2(a0, a1);
          sum = u.x + u.y;
        };
        // Against the running maximum while the others' maxima are on their
        // way (it stands unless the maximum moves); against the new maximum
        // on the first tile and when it moves.
        if (j > 0) exps(m);
        uint32_t mw[kSplit];
        if (!collect(mx_w, mw)) {
          ok = false;
          break;
        }
        float mxa = dec(mw[0]);
#pragma unroll
        for (int o = 1; o < kSplit; ++o) mxa = fmaxf(mxa, dec(mw[o]));
        const float m_new = (j == 0 || mxa > m + kLazyRescale) ? mxa : m;
        if (j == 0 || __any_sync(0xffffffffu, live && m_new != m)) exps(m_new);
#undef IKBO_S
        ptx::tc_fence_after();
        if (tr_t) trace_tile(p, k, 1, 4 * j + 2);
        const float alpha = fast_exp2(m - m_new);   // 0 on the first tile, 1 when m stays
        l = l * alpha + sum;
        // P (bf16 pairs) over the first half of this S buffer: the keys of
        // column group cg at columns cg * kCols / 2
        ptx::tmem_st(scol + cg * (kCols / 2), pk);
        ptx::tmem_st_wait();
        if (j > 0 && __any_sync(0xffffffffu, live && m_new != m)) {
          // O must hold exactly P_0..P_{j-1} V when it is rescaled: PV_{j-1}
          // complete (MMAs complete in order), PV_j not issued before p_full
          if (!pv_wait(gj - 1)) {
            ok = false;
            break;
          }
          const uint32_t ocol = tmem + lane_off + C::kOCol + cg * C::kPart;
#pragma unroll
          for (int c = 0; c < C::kOChunks; ++c) {
            uint32_t o[C::kOChunk];
            ptx::tmem_ld(ocol + c * C::kOChunk, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < C::kOChunk; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st(ocol + c * C::kOChunk, o);
          }
          ptx::tmem_st_wait();
        }
        m = m_new;
        ptx::tc_fence_before();
        __syncwarp();
        if (tr_t) trace_tile(p, k, 1, 4 * j + 3);
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl->p_full[sb]));
      }
      if (!ok) break;
      if (row == 0 && cg == 0) trace(p, k, kTrSmLastP);
      // ---- epilogue: the row sum goes out now, O is complete after the last PV
      const uint32_t l_w = publish(l);
      if (!pv_wait(g + n - 1)) break;
      if (row == 0 && cg == 0) trace(p, k, kTrEpiO);
      uint32_t lw[kSplit];
      if (!collect(l_w, lw)) break;
      // the row sum, added in group order by every thread of the row alike
      float lt = dec(lw[0]);
#pragma unroll
      for (int o = 1; o < kSplit; ++o) lt += dec(lw[o]);
      const bool tr_epi = row == 32 && cg == 0;    // epilogue timeline: one thread
      if (tr_epi) trace(p, k, kTrEpiSums);
      const uint32_t ocol = tmem + lane_off + C::kOCol + cg * C::kPart;
      // A split unit: each CTA of the pair finishes half of the rows (CTA 0
      // the first, CTA 1 the second) and sends the other half to its partner.
      const bool paired = w.unit >= 0;
      const int hrows = (rows + 1) >> 1;
      const bool mine = !paired || (cta_rank == 0 ? row < hrows : row >= hrows);
      const bool keep = live && mine;
      const bool send = live && !mine;
      const int vec0 = cg * C::kPart / 4;          // first 16-byte vector of this thread's columns
      if (__any_sync(0xffffffffu, send)) {
        // O / l and the log-sum-exp m + log2(l), straight into the partner's
        // Q buffers (rows of D fp32, 16-byte vectors swizzled by row)
        if (!W.warp_wait(ptx::smem_addr(&ctl->pair_go), 0, true)) break;
        const uint32_t peer = cta_rank ^ 1u;
        const uint32_t rbar = ptx::map_to_cta(ptx::smem_addr(&ctl->pair_recv), peer);
        const uint32_t rdst = ptx::map_to_cta(ptx::smem_addr(data), peer) + uint32_t(row * (D * 4));
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
        for (int cc = 0; cc < C::kOChunks; ++cc) {
          uint32_t o[C::kOChunk];
          ptx::tmem_ld(ocol + cc * C::kOChunk, o);
          ptx::tmem_ld_wait();
          if (send) {
#pragma unroll
            for (int q4 = 0; q4 < C::kOChunk / 4; ++q4) {
              const int vec = vec0 + cc * (C::kOChunk / 4) + q4;
              const float2 a = fmul2(make_float2(__uint_as_float(o[q4 * 4 + 0]), __uint_as_float(o[q4 * 4 + 1])), inv2);
              const float2 b2 = fmul2(make_float2(__uint_as_float(o[q4 * 4 + 2]), __uint_as_float(o[q4 * 4 + 3])), inv2);
              ptx::st_async_v4(rdst + uint32_t((vec ^ (row & 7)) * 16), a.x, a.y, b2.x, b2.y, rbar);
            }
          }
        }
        if (send && cg == 0)
          ptx::st_async_f32(ptx::map_to_cta(ptx::smem_addr(&ctl->partner_lse[row]), peer),
                            lt > 0.f ? m + fast_log2(lt) : -INFINITY, rbar);
        if (row == 0 && cg == 0) trace(p, k, kTrEpiStored);
        if (tr_epi) trace(p, k, kTrEpiSent);
      }
      if (__any_sync(0xffffffffu, keep)) {
        uint16_t* dst;
        if (w.q_row >= 0) {
          // a self-attention row: out_user[q_row + row, head, :]
          const int64_t srow = keep ? (int64_t)w.q_row + row : 0;
          dst = p.out_user + ((srow * p.H + w.head) * D) + cg * C::kPart;
        } else {
          const int ci = keep ? row / Lq : 0;
          const int tq = keep ? row - ci * Lq : 0;
          const int32_t gpos = w.cand_begin + ci;
          const int64_t cidx = keep ? (sorted ? gpos : perm[gpos]) : 0;
          dst = p.out + (((cidx * p.H + w.head) * (int64_t)Lq + tq) * D) + cg * C::kPart;
        }
        float lse_p = -INFINITY;
        if (paired) {
          // the partner's O / l and log-sum-exp for these rows
          if (!W.warp_wait(ptx::smem_addr(&ctl->pair_recv), 0, true)) break;
          if (row == 0 && cg == 0) trace(p, k, kTrArrived);
          if (keep) lse_p = ctl->partner_lse[row];
        }
        // out = (2^(m-M) O + 2^(lse_p-M) O_p / l_p) / (2^(m-M) l + 2^(lse_p-M))
        const float M = fmaxf(m, lse_p);
        const float a0 = fast_exp2(m - M), a1 = paired ? fast_exp2(lse_p - M) : 0.f;
        const float L = a0 * lt + a1;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float2 w0 = make_float2(a0 * inv, a0 * inv), w1 = make_float2(a1 * inv, a1 * inv);
#pragma unroll
        for (int cc = 0; cc < C::kOChunks; ++cc) {
          uint32_t o[C::kOChunk];
          ptx::tmem_ld(ocol + cc * C::kOChunk, o);
          ptx::tmem_ld_wait();
          if (keep) {
            float2 x[C::kOChunk / 2];
#pragma unroll
            for (int e = 0; e < C::kOChunk / 2; ++e)
              x[e] = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), w0);
            if (paired) {
#pragma unroll
              for (int q4 = 0; q4 < C::kOChunk / 4; ++q4) {
                const int vec = vec0 + cc * (C::kOChunk / 4) + q4;
                const float4 y = *reinterpret_cast<const float4*>(
                    data + row * (D * 4) + ((vec ^ (row & 7)) * 16));
                x[2 * q4] = fadd2(x[2 * q4], fmul2(make_float2(y.x, y.y), w1));
                x[2 * q4 + 1] = fadd2(x[2 * q4 + 1], fmul2(make_float2(y.z, y.w), w1));
              }
            }
            static_assert(C::kOChunk == 32, "32 columns per store");
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = pack_bf16(x[e].x, x[e].y);
            store_bf16x32(dst + cc * C::kOChunk, w);
          }
        }
        if (row == 0 && cg == 0) trace(p, k, paired ? kTrMerged : kTrEpiStored);
        if (tr_epi) trace(p, k, kTrEpiKept);
      }
      g += n;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  trace_pro(p, 9);
  // a leader that invited its partner's copy waits for it (bounded) before
  // its shared memory can go away, even if it gave up on the merge
  if (threadIdx.x == 0 && ctl->go_sent) W.drain(ptx::smem_addr(&ctl->pair_recv), 0);
  if (threadIdx.x == 0) trace(p, 0, kTrCtaEnd);
  __syncwarp();
  // Neither CTA of a pair may exit while the other can still touch its
  // memory.  The partner's copies complete on pair_recv, drained above; the
  // one other remote access, the producer's arrival on the partner's pair_go,
  // is ordered before this thread's barrier arrival by a fence (it may be
  // unconsumed if the partner gave up).  No other thread's memory operations
  // need ordering here, so the barrier itself is relaxed: it does not wait
  // for the epilogue's global stores.
  if (threadIdx.x == 0) ptx::fence_acq_rel_cluster();
  ptx::cluster_sync_relaxed();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
  trace_pro(p, 10);
}

}  // namespace ikbo
