// IKBO target attention, tcgen05 kernel with two query tiles of one user and
// head per work item, sharing one K/V stream.
//
// What it computes is what ikbo_attn_tc_kernel computes: the flash-attention
// forward of "Chapter 4: High-performance Kernels", §4.6.1, over the query
// tiles and user key ranges of "In-Kernel Broadcast Optimization", §3.1-§3.2.
// It is meant for users with many candidates (two or more query tiles per
// head), where the work is a dense contraction and the single-tile kernel
// leaves the tensor cores idle while the softmax of a tile runs.  Here the
// schedule is the ping-pong of "Optimizing Jagged Flash Attention with TLX",
// §2.1: two query tiles A and B (consecutive candidates of the same user, the
// same head) are in flight in one CTA, each with a softmax warpgroup of its
// own, and while one warpgroup turns its scores into weights the tensor cores
// work for the other.  Both tiles read the same K/V tile from shared memory,
// so each K/V tile is loaded once for up to 256 query rows: the IKBO saving of
// §3.1, twice over.
//
//   * tensor memory: S/P of A (128 columns), S/P of B, O of A and O of B
//     (D columns each);
//   * warp 0 (TMA producer, converged, one elected lane issuing): Q_A, K_0,
//     Q_B, then V_0, K_1, V_1, K_2, ...;
//   * warp 1 (MMA issuer, converged, one elected lane issuing): S_A(0),
//     S_B(0), then for every key tile j: PV_A(j), S_A(j+1), PV_B(j),
//     S_B(j+1).  S_A(j+1) overwrites the buffer that PV_A(j) reads P_A(j)
//     from, which is safe as the MMAs of one thread run in order; and
//     S_A(j+1) complete implies PV_A(j) complete, so the softmax may rescale
//     O_A as soon as it sees S_A(j+1);
//   * warps 4-7: softmax, correction and epilogue of tile A, warps 8-11 of
//     tile B, one thread per query row (all 128 key columns of a tile).
// An item whose user has an odd number of query tiles left has no tile B.
// When that query tile is the user's only one (no other item streams the
// same keys) and it has two key tiles or more, the planner marks it
// (n_split = 2) and its keys are split over the two warpgroups ("key-split"
// item): the query tile is loaded into both Q
// buffers, A takes key tiles 0, 2, 4, ..., B takes 1, 3, 5, ..., and the two
// partial results of every row are merged in the CTA with the log-sum-exp
// rule of "Chapter 4", §4.6.4 (each warpgroup finishes half of the output
// columns).  Its ring order is K0, K1, then per pair of key tiles (2i, 2i+1):
// V_2i, K_2i+2, V_2i+1, K_2i+3.  An item with one key tile and no tile B runs
// on warps 4-7 alone.  In a fused self + target call an item may also be two
// blocks of 128 rows of the user's own sequence (tile B the second block).
// Every wait is bounded, as in the single-tile kernel.
#pragma once

#include "ikbo_attn_tc.cuh"

namespace ikbo {

constexpr int kPpGroups = 2;                 // query tiles per item
constexpr int kPpSoftmaxWarps = 4;           // warps per tile: one thread per row

template <int D>
struct PpConfig {
  static constexpr int kCB = D / 64;
  static constexpr int kQBytes = kCB * kTileM * 128;
  static constexpr int kKVBytes = kCB * kBlockN * 128;
  static constexpr int kFit = (kDataBytes - kPpGroups * kQBytes) / kKVBytes;
  static constexpr int kSlots = kFit < kMaxSlots ? kFit : kMaxSlots;
  static constexpr int kTmemCols = 512;
  __host__ __device__ static constexpr uint32_t kSCol(int g) { return uint32_t(g) * kBlockN; }
  __host__ __device__ static constexpr uint32_t kOCol(int g) { return uint32_t(kPpGroups * kBlockN + g * D); }
  static_assert(kPpGroups * (kBlockN + D) <= kTmemCols, "TMEM budget");
  static_assert(kSlots >= 3, "ring size");
};

static_assert(kSoftmaxWarp0 + kPpGroups * kPpSoftmaxWarps == kTcThreads / 32, "warp roles");

// kSelf: a fused self + target call (items may be blocks of the user's own
// sequence); the target-only kernel carries none of that code.
template <int D, bool kSelf>
__global__ void __launch_bounds__(kTcThreads, 1)
ikbo_attn_pp_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap qmap1,
                    const __grid_constant__ CUtensorMap kmap_tmpl,
                    const __grid_constant__ CUtensorMap vmap_tmpl,
                    const __grid_constant__ CUtensorMap qumap) {
  using C = PpConfig<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* data = smem_raw;
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem_raw + kDataBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool layout_ok = (ptx::smem_addr(smem_raw) & 1023u) == 0;

  if (threadIdx.x == 0) {
    for (int g = 0; g < kPpGroups; ++g) {
      ptx::mbar_init(ptx::smem_addr(&ctl->q_full[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->q_empty[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[g]), kPpSoftmaxWarps);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_half[g]), kPpSoftmaxWarps);
      ptx::mbar_init(ptx::smem_addr(&ctl->pv_done[g]), 1);   // an item's last PV of tile g
    }
    for (int i = 0; i < kMaxSlots; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    // key-split items: both warpgroups published their row statistics, and
    // both finished reading the two accumulators (one arrival per warp)
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_go), kPpGroups * kPpSoftmaxWarps);
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_recv), kPpGroups * kPpSoftmaxWarps);
    // Cluster Launch Control: an answer arrived; the producer fills an item
    // queue slot; the MMA warp and the 8 softmax warps each release it
    ptx::mbar_init(ptx::smem_addr(&ctl->q.clc_bar), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->q.item_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->q.item_empty[i]), 1 + kPpGroups * kPpSoftmaxWarps);
    }
    ctl->abort_flag = 0;
    ctl->flags = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 2 && lane == 0) {
    if (p.n_cand > 0) ptx::prefetch_tensormap(&qmap);   // a self-only call encodes no Q map
    ptx::prefetch_tensormap(&kmap_tmpl);
    ptx::prefetch_tensormap(&vmap_tmpl);
    if (kSelf && p.q_user) ptx::prefetch_tensormap(&qumap);
  }
  // Cluster Launch Control: this SM's slot for the plan's tables and the
  // users' bounded V maps (one CTA per SM)
  const uint32_t sm = ptx::smid();
  const bool clc = !kSelf && p.clc && sm < (uint32_t)kClcSlots;
  uint8_t* slot = clc ? p.clc_slots + (size_t)sm * p.clc_slot_bytes : nullptr;
  if (p.fused && layout_ok) plan_load<16>(p, data);
  __syncthreads();
  if (!layout_ok || !p.fused || (!kSelf && p.clc && !clc)) {
    // this kernel plans in-kernel only; the host never launches it otherwise
    if (threadIdx.x == 0) {
      ctl->mode = kModeSkip;
      ctl->n_my_items = 0;
      ctl->sorted = 1;
      atomicOr(p.err_word, kErrLayout);
    }
  } else {
    plan_in_cta<!kSelf>(p, ctl, data, D, kPpGroups, reinterpret_cast<int32_t*>(slot));
    ptx::fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) ctl->bmaps_ready = 0;   // the planning's scan words are free now
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) trace_bounded(p, 0, kTrCtaStart);

  const uint32_t tmem = ctl->tmem_base;
  const int mode = ctl->mode;
  const int n_my = ctl->n_my_items;
  const bool sorted = ctl->sorted != 0;
  const int NS = C::kSlots;
  const int Lq = p.Lq;
  const int cpt = p.cands_per_tile;
  uint8_t* q_smem = data;
  uint8_t* kv_smem = data + kPpGroups * C::kQBytes;
  const int32_t* perm = p.perm_ws;
  const Waiter W{&ctl->abort_flag, p.err_word, p.timeout_ns};
  auto item_at = [&](int k) -> WorkItem {
    return k < kCtlItems ? ctl->items[k] : p.cta_items[(size_t)blockIdx.x * p.max_cta_items + k];
  };
  // Cluster Launch Control (mode kModeClc): the producer finds the CTA's k-th
  // unit and puts its item in queue slot k % 2 (ctl->items); the MMA and
  // softmax warps take it from there and release the slot when they start
  // item k + 1.  The plan's tables and the bounded V maps are in the SM's
  // slot.
  const bool dyn = mode == kModeClc;
  const int n_user_i = (int)p.n_user;
  const int32_t* tabs = reinterpret_cast<const int32_t*>(slot);
  CUtensorMap* user_maps = clc ? reinterpret_cast<CUtensorMap*>(slot + p.clc_map_offset) : nullptr;
  auto queue_release = [&](int k) {
    if (dyn && k > 0) ptx::mbar_arrive_warp(ptx::smem_addr(&ctl->q.item_empty[(k - 1) & 1]));
  };
  // the k-th item of a role's loop (false: none left, or a wait gave up)
  auto next_item = [&](int k, WorkItem& w, bool converged) -> bool {
    if (!dyn) {
      if (k >= n_my) return false;
      w = item_at(k);
      return true;
    }
    queue_release(k);
    const uint32_t bar = ptx::smem_addr(&ctl->q.item_full[k & 1]);
    if (!(converged ? W.conv_wait(bar, (k >> 1) & 1u) : W.warp_wait(bar, (k >> 1) & 1u))) return false;
    w = ctl->items[k & 1];
    return w.user >= 0;
  };
  auto ntiles = [](const WorkItem& w) { return ceil_div(w.kv_len, kBlockN); };
  // candidates of query tile g of an item (tile B holds those past the
  // first cpt); for a self-attention item (fused call), sequence rows (tile
  // B holds those past the first 128)
  auto tile_cands = [&](const WorkItem& w, int g) {
    const int per = (kSelf && w.q_row >= 0) ? kTileM : cpt;
    return g == 0 ? min(w.n_cand, per) : max(w.n_cand - per, 0);
  };
  // query rows of tile g
  auto tile_rows = [&](const WorkItem& w, int g) {
    return (kSelf && w.q_row >= 0) ? tile_cands(w, g) : tile_cands(w, g) * Lq;
  };
  // the user's only query tile, two key tiles or more: the keys split over
  // both warpgroups.  (A lone tile of a user with other tiles is not split:
  // its sibling items stream the same keys at one tile per step, and a split
  // item running ahead of them at two would fetch from DRAM what they then
  // fetch again: the sweeps ran 10-37 % slower so.)  At D = 64 the split is
  // not compiled: its code made every other item of the D = 64 sweeps 7 %
  // slower, while at D = 128 the same code made them 1.5-4 % faster.
  auto key_split = [&](const WorkItem& w) {
    return D == 128 && w.n_split == 2 && tile_cands(w, 1) == 0 && ntiles(w) >= 2;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // converged like the MMA warp: every lane waits, the elected lane issues
    // the loads (1-3 % faster than lane 0 alone in a divergent branch)
    if (mode != kModeSkip) {
      bool tail_ready = false;
      // K/V maps with an open row count; a tile reaching past row T goes
      // through a copy with the row count set to T (zero fill past the end)
      auto kv_map = [&](bool is_v, int32_t row) -> const void* {
        const int T = ctl->total_keys;
        // maps encoded with the row count T itself (a fused call states T)
        if ((kSelf && p.exact_rows) || row + kBlockN <= T)
          return is_v ? (const void*)&vmap_tmpl : (const void*)&kmap_tmpl;
        CUtensorMap* tail_k = p.map_slots + (size_t)p.map_stride * blockIdx.x;
        CUtensorMap* tail_v = tail_k + 1;
        if (!tail_ready) {
          if (lane == 0) {   // one lane writes the copies
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
              const uint4* s4 = reinterpret_cast<const uint4*>(mi == 0 ? &kmap_tmpl : &vmap_tmpl);
              uint4* d4 = reinterpret_cast<uint4*>(mi == 0 ? tail_k : tail_v);
#pragma unroll
              for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
              asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(d4),
                           "r"(T)
                           : "memory");
            }
            asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
          }
          __syncwarp();
          // every lane acquires them, whichever lane elect.sync picks to issue
          ptx::tensormap_acquire(tail_k);
          ptx::tensormap_acquire(tail_v);
          tail_ready = true;
        }
        return is_v ? (const void*)tail_v : (const void*)tail_k;
      };
      uint32_t kv_it = 0;
      uint32_t qn[kPpGroups] = {0, 0};
      // A user's partial last V tile goes through a copy of the V map bounded
      // at the user's end row (the TMA fills the other users' rows with
      // zeros), written by warp 2 after planning: one per item, or with
      // Cluster Launch Control one per user.
      bool bm_ready = false;
      int cur_item = 0, cur_user = 0;
      auto v_map_for = [&](int32_t row, int32_t end) -> const void* {
        if (row + kBlockN <= end) return kv_map(true, row);
        if (!bm_ready) {
          bool got = true;
          if (lane == 0) got = wait_bounded_maps(p, ctl);
          if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) return nullptr;
          bm_ready = true;
        }
        CUtensorMap* m = dyn ? user_maps + cur_user
                             : p.map_slots + (size_t)p.map_stride * blockIdx.x + 2 + cur_item;
        ptx::tensormap_acquire(m);
        ptx::prefetch_tensormap(m);
        return m;
      };
      // the next ring load: one K or V tile (128 keys x D of one head); the
      // item's keys end at row `end`
      auto ring = [&](bool is_v, int head, int32_t row, int32_t end) -> bool {
        const uint32_t slot = kv_it % NS;
        // the map first: a bounded map's acquire and descriptor fetch then
        // overlap the wait for the slot
        const void* map = is_v ? v_map_for(row, end) : kv_map(false, row);
        if (!map) return false;
        if (!W.conv_wait(ptx::smem_addr(&ctl->kv_empty[slot]), ((kv_it / NS) & 1u) ^ 1u)) return false;
        const uint32_t bar = ptx::smem_addr(&ctl->kv_full[slot]);
        const uint32_t dst = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
        ptx::mbar_arrive_expect_tx_warp(bar, C::kKVBytes);
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb)
          ptx::tma_load_2d_warp(dst + cb * kBlockN * 128, map, bar, head * D + cb * 64, row);
        ++kv_it;
        return true;
      };
      // query tile src of item w into Q buffer g
      auto load_q = [&](int g, const WorkItem& w, int src) -> bool {
        if (!W.conv_wait(ptx::smem_addr(&ctl->q_empty[g]), (qn[g] & 1u) ^ 1u)) return false;
        ++qn[g];
        if (p.debug_flags & 1) return true;    // test hook: never arm the Q barrier
        const int nc = tile_cands(w, src);
        const int32_t c0 = w.cand_begin + src * cpt;
        const uint32_t qbar = ptx::smem_addr(&ctl->q_full[g]);
        const uint32_t qdst = ptx::smem_addr(q_smem + g * C::kQBytes);
        if (kSelf && w.q_row >= 0) {
          // 128 rows of the user sequence's queries (rows past T read as zeros)
          ptx::mbar_arrive_expect_tx_warp(qbar, uint32_t(C::kCB * kTileM * 128));
          for (int cb = 0; cb < C::kCB; ++cb)
            ptx::tma_load_2d_warp(qdst + cb * kTileM * 128, &qumap, qbar, w.head * D + cb * 64,
                                  w.q_row + src * kTileM);
        } else if (sorted) {
          const int nb = p.qbox;
          const int nbox = ceil_div(nc, nb);
          ptx::mbar_arrive_expect_tx_warp(qbar, uint32_t(nbox * nb * Lq * 128 * C::kCB));
          for (int cb = 0; cb < C::kCB; ++cb)
            for (int bx = 0; bx < nbox; ++bx)
              ptx::tma_load_4d_warp(qdst + cb * kTileM * 128 + bx * nb * Lq * 128, &qmap, qbar, cb * 64, 0, w.head,
                               c0 + bx * nb);
        } else {
          ptx::mbar_arrive_expect_tx_warp(qbar, uint32_t(nc * Lq * 128 * C::kCB));
          for (int i = 0; i < nc; ++i) {
            const int32_t c = perm[c0 + i];
            for (int cb = 0; cb < C::kCB; ++cb)
              ptx::tma_load_4d_warp(qdst + cb * kTileM * 128 + i * Lq * 128, &qmap1, qbar, cb * 64, 0, w.head, c);
          }
        }
        return true;
      };
      // Cluster Launch Control: the CTA's first unit is its own index; each
      // next one is the index of a CTA of the grid that has not started,
      // which the hardware cancels at this CTA's request.  At D = 128 the
      // request goes out once the current unit's loads are all issued: its
      // answer still arrives while the unit's last key tiles are computed,
      // and the unit taken is the next in the list when this CTA is nearly
      // free.  (Asked at the start of the current unit, the CTAs that
      // started the longest units took the next-longest at once: on
      // odd_groups_2048x16 the busiest CTA ran 30 % above the mean.)  At
      // D = 64 the late request made every unit slower (2 % on the sweeps;
      // asking a few loads earlier did not help either), so there it goes
      // out as the unit starts.
      // The grid is sized by a bound on the units: indices past the plan's
      // count are taken over too, and skipped, until a request cancels
      // nothing.
      constexpr bool kLateAsk = D == 128;
      const int N = ctl->n_units;
      const uint32_t clc_bar = ptx::smem_addr(&ctl->q.clc_bar), clc_resp = ptx::smem_addr(ctl->q.clc_resp);
      uint32_t clc_phase = 0;
      bool clc_pending = false;
      auto clc_ask = [&]() {
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(clc_bar, 16);
          ptx::clc_try_cancel(clc_resp, clc_bar);
        }
        clc_pending = true;
      };
      auto clc_next = [&](int k) -> int {
        if (k == 0) {
          if ((int)blockIdx.x >= N) return -1;   // no unit of its own, none after it either
          if (!kLateAsk) clc_ask();
          return (int)blockIdx.x;
        }
        while (clc_pending) {
          if (!W.conv_wait(clc_bar, clc_phase & 1u)) return -1;   // (still pending: drained below)
          ++clc_phase;
          clc_pending = false;
          uint32_t x = 0;
          if (!ptx::clc_query(clc_resp, x)) return -1;   // nothing left to take over
          if (!kLateAsk || (int)x >= N) clc_ask();
          if ((int)x < N) return (int)x;
        }
        return -1;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (dyn) {
          // the next unit (once queue slot k % 2 is free), as the slot's item
          if (k >= 2 && !W.conv_wait(ptx::smem_addr(&ctl->q.item_empty[k & 1]), ((k >> 1) - 1) & 1u)) break;
          const int unit = clc_next(k);
          if (lane == 0) {
            WorkItem x;
            if (unit >= 0) {
              const int n1 = n_user_i + 1;
              decode_unit(unit, tabs, tabs + n1, tabs + 2 * n1, tabs + 3 * n1, n_user_i, kPpGroups, cpt,
                          false, x);
            } else {
              x.user = -1;   // no unit left: the roles stop
            }
            ctl->items[k & 1] = x;
            ptx::mbar_arrive(ptx::smem_addr(&ctl->q.item_full[k & 1]));
          }
          __syncwarp();
          w = ctl->items[k & 1];
          if (w.user < 0) break;
        } else if (!next_item(k, w, true)) {
          break;
        }
        cur_item = k;
        cur_user = w.user;
        const int n = ntiles(w);
        const bool has_b = tile_cands(w, 1) > 0;
        if (lane == 0) trace_bounded(p, k, kTrProdItem);
        // Q_A and K_0 first: S_A(0) needs only these
        const int32_t end = w.kv_begin + w.kv_len;
        if (!key_split(w)) {
          ok = load_q(0, w, 0) && ring(false, w.head, w.kv_begin, end) && (!has_b || load_q(1, w, 1));
          for (int j = 0; j < n && ok; ++j) {
            ok = ring(true, w.head, w.kv_begin + j * kBlockN, end);
            if (ok && j + 1 < n) ok = ring(false, w.head, w.kv_begin + (j + 1) * kBlockN, end);
          }
        } else {
          // the same query tile into both buffers; K0 for A, K1 for B, then
          // per pair of key tiles V_2i, K_2i+2, V_2i+1, K_2i+3 (the MMA order)
          auto row_of = [&](int t) { return w.kv_begin + t * kBlockN; };
          ok = load_q(0, w, 0) && ring(false, w.head, row_of(0), end) && load_q(1, w, 0) &&
               ring(false, w.head, row_of(1), end);
          for (int t = 0; t < n && ok; t += 2) {
            ok = ring(true, w.head, row_of(t), end);
            if (ok && t + 2 < n) ok = ring(false, w.head, row_of(t + 2), end);
            if (ok && t + 1 < n) ok = ring(true, w.head, row_of(t + 1), end);
            if (ok && t + 3 < n) ok = ring(false, w.head, row_of(t + 3), end);
          }
        }
        if (lane == 0) trace_bounded(p, k, kTrProdIssued);
        if (kLateAsk && dyn && ok) clc_ask();   // the next unit
      }
      // Drain: every armed barrier phase must complete before the CTA exits
      // (a cancellation request still out after an abort included).
      if (lane == 0 && clc_pending) W.drain(clc_bar, clc_phase & 1u);
      if (lane == 0)
      for (uint32_t s = 0; s < (uint32_t)NS && s < kv_it; ++s) {
        const uint32_t uses = (kv_it - s + NS - 1) / NS;
        W.drain(ptx::smem_addr(&ctl->kv_full[s]), (uses - 1) & 1u);
      }
      if (lane == 0 && !(p.debug_flags & 1))
        for (int g = 0; g < kPpGroups; ++g)
          if (qn[g]) W.drain(ptx::smem_addr(&ctl->q_full[g]), (qn[g] - 1) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // The whole warp runs this loop, converged (waits included), and the
    // elected lane issues every MMA and commit.
    if (mode != kModeSkip) {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kTileM, kBlockN, 0);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kTileM, D, 1);
      uint32_t kv_base = 0;                       // ring index of the item's K_0
      uint32_t qn[kPpGroups] = {0, 0}, pn[kPpGroups] = {0, 0};
      auto kv_ready = [&](uint32_t idx) -> bool {
        if (!W.conv_wait(ptx::smem_addr(&ctl->kv_full[idx % NS]), (idx / NS) & 1u)) return false;
        ptx::tc_fence_after();
        return true;
      };
      // S_g = Q_g K^T, K in ring slot kslot, into S buffer g
      auto issue_s = [&](int g, uint32_t kslot) {
        const uint32_t q_base = ptx::smem_addr(q_smem + g * C::kQBytes);
        const uint32_t k_base = ptx::smem_addr(kv_smem + kslot * C::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int cb = kk >> 2;
          const uint32_t koff = (kk & 3) * 32;
          const uint64_t a = ptx::smem_desc_sw128(q_base + cb * kTileM * 128 + koff, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(k_base + cb * kBlockN * 128 + koff, 16, 1024);
          ptx::mma_ss_warp(tmem + C::kSCol(g), a, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_warp(ptx::smem_addr(&ctl->s_full[g]));
      };
      // O_g += P_g V over keys [64 h, 64 h + 64) of the tile, P from the
      // first 64 columns of S buffer g, V (MN-major) in ring slot vslot
      auto issue_pv_half = [&](int g, uint32_t vslot, int h, bool acc) {
        const uint32_t v_base = ptx::smem_addr(kv_smem + vslot * C::kKVBytes);
#pragma unroll
        for (int q = 0; q < kBlockN / 32; ++q) {
          const int kk = h * (kBlockN / 32) + q;
          const uint64_t bdesc = ptx::smem_desc_sw128(v_base + kk * 16 * 128, kBlockN * 128, 1024);
          ptx::mma_ts_warp(tmem + C::kOCol(g), tmem + C::kSCol(g) + kk * 8, bdesc, kIdescPV,
                      (acc || kk > 0) ? 1u : 0u);
        }
      };
      // P_g of the current tile: first half (h = 0) or all of it (h = 1);
      // one phase of each barrier per tile
      auto p_ready = [&](int g, int h) -> bool {
        if (!W.conv_wait(ptx::smem_addr(h == 0 ? &ctl->p_half[g] : &ctl->p_full[g]), pn[g] & 1u)) return false;
        if (h == 1) ++pn[g];
        ptx::tc_fence_after();
        return true;
      };
      // O_g += P_g V_j: each half once the softmax has written it
      auto issue_pv = [&](int g, uint32_t vslot, bool acc) -> bool {
        if (!p_ready(g, 0)) return false;
        issue_pv_half(g, vslot, 0, acc);
        if (!p_ready(g, 1)) return false;
        issue_pv_half(g, vslot, 1, true);
        return true;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        WorkItem w;
        if (!next_item(k, w, true)) break;
        const int n = ntiles(w);
        const bool has_b = tile_cands(w, 1) > 0;
        const bool split = key_split(w);
        if (!W.conv_wait(ptx::smem_addr(&ctl->q_full[0]), qn[0] & 1u)) break;
        if ((has_b || split) && !W.conv_wait(ptx::smem_addr(&ctl->q_full[1]), qn[1] & 1u)) break;
        ptx::tc_fence_after();
        if (lane == 0) trace_bounded(p, k, kTrMmaQ);
        if (split) {
          // A on key tiles 0, 2, 4, ..., B on 1, 3, 5, ...: per pair of key
          // tiles PV_A, S_A(next), PV_B, S_B(next), the ring consumed in order
          const int na = (n + 1) / 2, nb = n / 2;
          uint32_t ri = kv_base;
          // S_g on the K tile at ring index ri; the last S_g of the item frees Q_g
          auto s_at = [&](int g, bool last) -> bool {
            if (!kv_ready(ri)) return false;
            issue_s(g, ri % NS);
            if (last) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[g]));
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[ri % NS]));
            ++ri;
            return true;
          };
          // O_g += P_g V for the V tile at ring index ri; the last one marks O_g complete
          auto pv_at = [&](int g, bool acc, bool last) -> bool {
            if (!kv_ready(ri) || !issue_pv(g, ri % NS, acc)) return false;
            if (last) ptx::mma_commit_warp(ptx::smem_addr(&ctl->pv_done[g]));
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[ri % NS]));
            ++ri;
            return true;
          };
          ok = s_at(0, na == 1) && s_at(1, nb == 1);
          if (ok && lane == 0) trace_bounded(p, k, kTrMmaFirstS);
          for (int j = 0; j < na && ok; ++j) {
            ok = pv_at(0, j > 0, j + 1 == na);
            if (ok && j + 1 < na) ok = s_at(0, j + 2 == na);
            if (ok && j < nb) ok = pv_at(1, j > 0, j + 1 == nb);
            if (ok && j + 1 < nb) ok = s_at(1, j + 2 == nb);
          }
          if (!ok) break;
          if (lane == 0) trace_bounded(p, k, kTrMmaLastPV);
          kv_base = ri;
          ++qn[0];
          ++qn[1];
          continue;
        }
        if (!kv_ready(kv_base)) break;
        {
          const uint32_t ks = kv_base % NS;
          issue_s(0, ks);
          if (n == 1) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[0]));
          if (has_b) {
            issue_s(1, ks);
            if (n == 1) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[1]));
          }
          ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[ks]));
        }
        if (lane == 0) trace_bounded(p, k, kTrMmaFirstS);
        for (int j = 0; j < n; ++j) {
          const uint32_t vi = kv_base + 2 * j + 1, ki = vi + 1;
          const bool more = j + 1 < n;
          if (!kv_ready(vi) || !issue_pv(0, vi % NS, j > 0)) {
            ok = false;
            break;
          }
          if (!more) ptx::mma_commit_warp(ptx::smem_addr(&ctl->pv_done[0]));
          if (more) {
            if (!kv_ready(ki)) {
              ok = false;
              break;
            }
            issue_s(0, ki % NS);
            if (j + 2 == n) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[0]));
          }
          if (has_b) {
            if (!issue_pv(1, vi % NS, j > 0)) {
              ok = false;
              break;
            }
            if (!more) ptx::mma_commit_warp(ptx::smem_addr(&ctl->pv_done[1]));
          }
          ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[vi % NS]));
          if (more) {
            if (has_b) {
              issue_s(1, ki % NS);
              if (j + 2 == n) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[1]));
            }
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[ki % NS]));
          }
        }
        if (lane == 0) trace_bounded(p, k, kTrMmaLastPV);
        kv_base += 2 * n;
        ++qn[0];
        if (has_b) ++qn[1];
      }
      // All issued MMAs must finish before tensor memory is released.
      ptx::mma_commit_warp(ptx::smem_addr(&ctl->drain));
      if (lane == 0) W.drain(ptx::smem_addr(&ctl->drain), 0);
    }
    __syncwarp();
  } else if ((warp == 2 || warp == 3) && mode != kModeSkip) {
    prefetch_v_late(p, ctl->total_keys, D);
    if (warp == 2) {
      if (dyn)
        write_user_maps(ctl, user_maps, &vmap_tmpl, tabs, tabs + n_user_i + 1, n_user_i);
      else
        write_bounded_maps(p, ctl, &vmap_tmpl, n_my, item_at);
    }
  } else if (warp >= kSoftmaxWarp0 && mode != kModeSkip) {
    // ------------------------------------------- softmax / correction / epilogue
    const int g = (warp - kSoftmaxWarp0) / kPpSoftmaxWarps;   // query tile of this warp
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                      // TMEM lane == tile row
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t scol = tmem + lane_off + C::kSCol(g);
    const uint32_t ocol = tmem + lane_off + C::kOCol(g);
    const float sl2 = p.scale_log2;
    uint32_t tn = 0, dn = 0;                                  // S tiles and items of this tile so far
    uint32_t sp = 0;                                          // key-split items so far
    for (int k = 0;; ++k) {
      WorkItem w;
      if (!next_item(k, w, false)) break;
      const bool split = key_split(w);
      const int tg = split ? 0 : g;                           // the query tile whose rows these are
      const int nc = tile_cands(w, tg);
      if (nc == 0) continue;
      const int n = ntiles(w);
      const int ng = split ? (n - g + 1) / 2 : n;             // key tiles of this warpgroup
      // Rows past the tile's queries hold stale shared memory; their results
      // are never stored, and they are left out of every decision below.
      const bool live = row < tile_rows(w, tg);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < ng; ++j, ++tn) {
        if (!W.warp_wait(ptx::smem_addr(&ctl->s_full[g]), tn & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // All 128 scores of the row at once (one TMEM round trip); P is
        // written over them in place, two keys per 32-bit word.
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(scol + c * 32, r[c]);
        ptx::tmem_ld_wait();
#define IKBO_R(e) __uint_as_float(r[(e) >> 5][(e) & 31])
        // Scores enter the exponent as fma(s, sc, -m): raw scores with
        // sc = scale on full tiles for scale > 0 (their order is that of the
        // scaled ones), else scaled here with the keys past the user's
        // sequence at -inf (sc = 1).
        const int valid = min(kBlockN, w.kv_len - (split ? 2 * j + g : j) * kBlockN);
        float sc = sl2;
        if (valid < kBlockN || !(sl2 > 0.f)) {
#pragma unroll
          for (int e = 0; e < kBlockN; ++e) {
            const float tt = IKBO_R(e) * sl2;
            r[e >> 5][e & 31] = __float_as_uint(e < valid ? tt : -INFINITY);
          }
          sc = 1.f;
        }
        float mx;
        {
          // four independent chains
          float a0 = fmaxf(IKBO_R(0), IKBO_R(1)), a1 = fmaxf(IKBO_R(2), IKBO_R(3));
          float a2 = fmaxf(IKBO_R(4), IKBO_R(5)), a3 = fmaxf(IKBO_R(6), IKBO_R(7));
#pragma unroll
          for (int e = 8; e < kBlockN; e += 8) {
            a0 = fmax3(a0, IKBO_R(e), IKBO_R(e + 1));
            a1 = fmax3(a1, IKBO_R(e + 2), IKBO_R(e + 3));
            a2 = fmax3(a2, IKBO_R(e + 4), IKBO_R(e + 5));
            a3 = fmax3(a3, IKBO_R(e + 6), IKBO_R(e + 7));
          }
          mx = fmax3(a0, a1, fmaxf(a2, a3)) * sc;
        }
        // The running maximum moves only when the tile's exceeds it by more
        // than kLazyRescale (weights stay <= 2^8), and always on an item's
        // first tile.
        const float m_new = (j == 0 || mx > m + kLazyRescale) ? mx : m;
        const float alpha = fast_exp2(m - m_new);   // 0 on the first tile, 1 when m stays
        if (j > 0 && __any_sync(0xffffffffu, live && m_new != m)) {
          // O must hold exactly P_0..P_{j-1} V when it is rescaled: S_g(j)
          // complete implies PV_g(j-1) complete (issued before it), and
          // PV_g(j) waits for this tile's P
          // (16 columns at a time: the scores are live in registers here)
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            ptx::tmem_ld16(ocol + c * 16, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st16(ocol + c * 16, o);
          }
        }
        // P = 2^(s sc - m_new) as bf16 pairs, key pair e / 2 into word e / 2
        // (a word whose scores were read already), in two halves of 64 keys:
        // the MMA warp starts O += P V on the first while the second is made.
        float sum = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 sc2 = make_float2(sc, sc), nr2 = make_float2(-m_new, -m_new);
          float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 64 * h; e < 64 * h + 64; e += 2) {
            const float2 x = ffma2(make_float2(IKBO_R(e), IKBO_R(e + 1)), sc2, nr2);
            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            if ((e >> 1) & 1) a1 = fadd2(a1, pe); else a0 = fadd2(a0, pe);
            r[e >> 6][(e >> 1) & 31] = pack_bf16(pe.x, pe.y);
          }
          const float2 u = fadd2(a0, a1);
          sum += u.x + u.y;
          ptx::tc_fence_before();
          ptx::tmem_st32(scol + 32 * h, r[h]);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          ptx::mbar_arrive_warp(ptx::smem_addr(h == 0 ? &ctl->p_half[g] : &ctl->p_full[g]));
        }
#undef IKBO_R
        l = l * alpha + sum;
        m = m_new;
      }
      if (!ok) break;
      // ---- epilogue: O after the item's last PV of this tile
      if (!W.warp_wait(ptx::smem_addr(&ctl->pv_done[g]), dn & 1u)) break;
      ++dn;
      ptx::tc_fence_after();
      if (row == 0 && g == 0) trace_bounded(p, k, kTrEpiO);
      uint16_t* dst;
      if (kSelf && w.q_row >= 0) {
        // a self-attention row: out_user[q_row + 128 tg + row, head, :]
        const int64_t srow = live ? (int64_t)w.q_row + tg * kTileM + row : 0;
        dst = p.out_user + ((srow * p.H + w.head) * D);
      } else {
        const int ci = live ? row / Lq : 0;
        const int tq = live ? row - ci * Lq : 0;
        const int32_t gpos = w.cand_begin + tg * cpt + ci;
        const int64_t cidx = live ? (sorted ? gpos : perm[gpos]) : 0;
        dst = p.out + (((cidx * p.H + w.head) * (int64_t)Lq + tq) * D);
      }
      if (split) {
        // Merge the two warpgroups' partial results of this row ("Chapter 4",
        // §4.6.4): with M = max(m_A, m_B), a = 2^(m_A - M), b = 2^(m_B - M),
        // out = (a O_A + b O_B) / (a l_A + b l_B).  Each warpgroup finishes
        // half of the columns, reading both accumulators.
        ctl->ab_ml[g][row] = make_float2(m, l);
        __syncwarp();
        ptx::mbar_arrive_warp(ptx::smem_addr(&ctl->pair_go));
        if (!W.warp_wait(ptx::smem_addr(&ctl->pair_go), sp & 1u)) break;
        const float2 other = ctl->ab_ml[g ^ 1][row];
        const float mm = fmaxf(m, other.x);
        const float a = fast_exp2(m - mm), b = fast_exp2(other.x - mm);
        const float den = a * l + b * other.y;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const float2 fa2 = make_float2(a * inv, a * inv), fb2 = make_float2(b * inv, b * inv);
        const uint32_t own = ocol, oth = tmem + lane_off + C::kOCol(g ^ 1);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int col = g * (D / 2) + c * 32;
          uint32_t oa[32], ob[32];
          ptx::tmem_ld32(own + col, oa);
          ptx::tmem_ld32(oth + col, ob);
          ptx::tmem_ld_wait();
          if (live) {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x = ffma2(make_float2(__uint_as_float(oa[2 * e]), __uint_as_float(oa[2 * e + 1])), fa2,
                                     fmul2(make_float2(__uint_as_float(ob[2 * e]), __uint_as_float(ob[2 * e + 1])), fb2));
              w[e] = pack_bf16(x.x, x.y);
            }
            store_bf16x32(dst + col, w);
          }
        }
        if (row == 0 && g == 0) trace_bounded(p, k, kTrEpiStored);
        // both warpgroups are done with both accumulators (and with the row
        // statistics) before either hands over the next item's first P
        ptx::tc_fence_before();
        __syncwarp();
        ptx::mbar_arrive_warp(ptx::smem_addr(&ctl->pair_recv));
        if (!W.warp_wait(ptx::smem_addr(&ctl->pair_recv), sp & 1u)) break;
        ++sp;
        continue;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(ocol + c * 32, o);
        ptx::tmem_ld_wait();
        if (live) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), inv2);
            w[e] = pack_bf16(x.x, x.y);
          }
          store_bf16x32(dst + c * 32, w);
        }
      }
      if (row == 0 && g == 0) trace_bounded(p, k, kTrEpiStored);
      // the next item's PV_g(0) overwrites O_g: it waits for that item's
      // first P of this tile, which these warps hand over only after the
      // reads above
      ptx::tc_fence_before();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_bounded(p, 0, kTrCtaEnd);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace ikbo
