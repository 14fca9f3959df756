// IKBO target attention, tcgen05 kernel for batches of few work units: the
// key tiles of one query tile interleaved over two softmax warpgroups.
//
// What it computes is what ikbo_attn_tc_kernel computes: the flash-attention
// forward of "Chapter 4: High-performance Kernels", §4.6.1, over the query
// tiles and user key ranges of "In-Kernel Broadcast Optimization", §3.1-§3.2
// (a query tile holds up to 128 rows of candidates of ONE user; each K/V tile
// is loaded once for all of them).
//
// It is meant for the pages' own shape: ~70 candidates per user (§1.1), so one
// query tile per user and head, and fewer (user, head, query tile) units than
// SMs.  A unit's time is then its chain of key tiles, so each CTA takes one
// unit and deals its key tiles to two softmax warpgroups in turn: A takes
// tiles 0, 2, 4, ..., B tiles 1, 3, 5, ..., each with an S buffer and an O
// accumulator of its own in tensor memory and a P buffer in shared memory,
// so the softmax of two tiles runs at once.  Both read the same Q tile.  P
// is written to shared memory (the A operand of an SS-form P.V MMA), so a
// warpgroup's S buffer is free as soon as its scores are in registers, and
// the MMA warp computes its next S while it works on the current one.  At
// the end the two partial results of every row are merged in the CTA with
// the log-sum-exp rule of "Chapter 4", §4.6.4 (Flash-Decoding): with
// M = max(m_A, m_B), a = 2^(m_A - M), b = 2^(m_B - M),
// out = (a O_A + b O_B) / (a l_A + b l_B).
//
// A unit whose key tiles exceed a CTA's balanced share by far (one user with
// tens of thousands of keys) is cut into chunks of consecutive key tiles on
// several CTAs, when every chunk still gets a CTA of its own.  Every chunk
// but the first writes O / l and its log-sum-exp to global memory and raises
// a flag; the first chunk's CTA waits for the flags (bounded), merges by the
// same rule and stores the rows.  All CTAs of the launch are resident at
// once (one per SM, grid = SMs), so such a wait always ends; a unit is never
// cut into chunks of one CTA.  The flags carry a value unique to the call and
// are reset by the merging CTA.
//
// With more units than CTAs, units are dealt to CTAs in boustrophedon order
// over the users sorted by key tiles, longest first ("Optimizing Jagged Flash
// Attention with TLX", §2.2), and each CTA runs its units in turn.
//
// Warp roles (384 threads):
//   warp 0      TMA producer (converged, one elected lane issues): the Q tile,
//               then K0, K1, K2, K3, V0, V1, K4, K5, V2, V3, ... into a ring;
//   warp 1      TMEM owner and MMA issuer (converged): S_A = Q K0^T,
//               S_B = Q K1^T, then per pair of key tiles (2i, 2i + 1), with
//               g = j % 2: S_g = Q K_(j+2)^T once warpgroup g has read its
//               scores of tile j, then O_g += P_g V_j once it has written P_g.
//               The ring is consumed strictly in order;
//   warp 2      writes the bounded V maps of the CTA's items (see
//               write_bounded_maps); warp 3 has no role;
//   warps 4-7   softmax, correction and epilogue of warpgroup A, one thread
//               per query row (TMEM lane), all 128 keys of a tile;
//   warps 8-11  the same for warpgroup B.
// The last key tile of a user may reach into the next users' rows: its V
// tile is loaded through a map bounded at the user's end row, so those rows
// arrive as zeros (see write_bounded_map).  Every wait is bounded.
#pragma once

#include "ikbo_attn_tc.cuh"

namespace ikbo {

constexpr int kAbGroups = 2;          // softmax warpgroups: even and odd key tiles
constexpr int kAbMaxSplit = 8;        // key-range chunks of one unit at most
// A unit is cut into chunks only when its key tiles exceed the balanced
// share of a CTA by more than this: the merge through global memory costs
// a few microseconds, several tiles' worth.
constexpr int kAbSplitSlack = 6;

template <int D>
struct AbConfig {
  static constexpr int kCB = D / 64;
  static constexpr int kQBytes = kCB * kTileM * 128;
  static constexpr int kKVBytes = kCB * kBlockN * 128;
  static constexpr int kQBufs = 1;
  static constexpr int kPBytes = kTileM * kBlockN * 2;   // P of one warpgroup: 128 rows x 128 keys, bf16
  static constexpr int kFit = (kDataBytes - kQBufs * kQBytes - kAbGroups * kPBytes) / kKVBytes;
  static constexpr int kSlots = kFit < kMaxSlots ? kFit : kMaxSlots;
  static constexpr int kTmemCols = 512;
  static constexpr int kHalf = D / 2;   // output columns each warpgroup finishes
  __host__ __device__ static constexpr uint32_t kSCol(int g) { return uint32_t(g) * kBlockN; }
  __host__ __device__ static constexpr uint32_t kOCol(int g) { return uint32_t(kAbGroups * kBlockN + g * D); }
  static_assert(kAbGroups * (kBlockN + D) <= kTmemCols, "TMEM budget");
  static_assert(kSlots >= 3, "ring size");
};

static_assert(kSoftmaxWarp0 + 4 * kAbGroups == kTcThreads / 32, "warp roles");

// Exclusive prefix over users of f(u), users taken in rank order (order[rank]
// when lpt, else the index): ubefore[rank], and the total in ubefore[n_user]
// and ctl->ab_units.  All threads of the CTA call it; it ends with a barrier.
template <typename F>
__device__ void ab_user_prefix(TcCtrl* ctl, int32_t* ubefore, const int32_t* order, bool lpt,
                               int n_user, F f) {
  const int tid = threadIdx.x, nt = blockDim.x;
  __syncthreads();   // every thread has read the previous prefix and total
  if (n_user <= 32) {
    if (tid < 32) {
      const int x = tid < n_user ? f(lpt ? order[tid] : tid) : 0;
      int v = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (tid >= o) v += y;
      }
      if (tid < n_user) ubefore[tid] = v - x;
      if (tid == 31) {
        ubefore[n_user] = v;
        ctl->ab_units = v;
      }
    }
  } else {
    int carry = 0;
    for (int base = 0; base < n_user; base += nt) {
      const int rk = base + tid;
      const int x = rk < n_user ? f(lpt ? order[rk] : rk) : 0;
      int tot;
      const int ex = block_scan_excl(x, ctl->red, &tot);
      if (rk < n_user) ubefore[rk] = carry + ex;
      carry += tot;
    }
    if (tid == 0) {
      ubefore[n_user] = carry;
      ctl->ab_units = carry;
    }
  }
  __syncthreads();
}

// Work items of this CTA (after plan_group), all threads.  Per user u: key
// tiles n_u = ceil(L_u / 128), query tiles q_u = ceil(r_u / cands per tile)
// (0 without candidates or keys), units H q_u.
//   * units <= CTAs: CTA i takes unit i.  With c = ceil(W / CTAs), W the key
//     tiles of all units, a unit with n_u > c + kAbSplitSlack is cut into
//     s_u = min(kAbMaxSplit, ceil(n_u / c)) chunks of consecutive key tiles,
//     provided the chunks of all units still fit the CTAs; chunk i on CTA i.
//   * more units: boustrophedon dealing over users sorted longest first.
// Returns the units (or chunks) in all.
__device__ int plan_ab(const AttnParams& p, TcCtrl* ctl, uint8_t* scratch) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int grid = gridDim.x, b = blockIdx.x;
  const int n_cand = (int)p.n_cand, n_user = (int)p.n_user;
  PlanScratch S(scratch, n_user, n_cand);
  const int32_t* const off = S.off;
  const int32_t* const cs = S.cs;
  int32_t* const order = S.order;
  int32_t* const ubefore = S.ubefore;
  const int cpt = p.cands_per_tile;
  const int H = p.H;
  auto tiles_of = [&](int u) { return ceil_div(off[u + 1] - off[u], kBlockN); };
  auto qtiles_of = [&](int u) {
    const int r = cs[u + 1] - cs[u], L = off[u + 1] - off[u];
    return (r > 0 && L > 0) ? ceil_div(r, cpt) : 0;
  };
  // chunks of a unit of user u for chunk size c (0: no unit is cut)
  auto splits_of = [&](int u, int c) {
    const int n = tiles_of(u);
    return (c > 0 && n > c + kAbSplitSlack) ? min(kAbMaxSplit, ceil_div(n, c)) : 1;
  };
  ab_user_prefix(ctl, ubefore, order, false, n_user, [&](int u) { return H * qtiles_of(u); });
  trace_pro(p, 2);
  const int U = ctl->ab_units;
  int c = 0;
  int n_units = U;
  bool lpt = false;
  if (U <= grid) {
    // the key tiles of all units (a unit's counted up to 2^16, enough for the decision)
    ab_user_prefix(ctl, ubefore, order, false, n_user,
                   [&](int u) { return H * qtiles_of(u) * min(tiles_of(u), 1 << 16); });
    const int W = ctl->ab_units;
    c = max(1, ceil_div(W, grid));
    ab_user_prefix(ctl, ubefore, order, false, n_user,
                   [&](int u) { return H * qtiles_of(u) * splits_of(u, c); });
    n_units = ctl->ab_units;
    if (n_units > grid || n_units == U) {
      // no unit is cut (the chunks would not all get a CTA, or none needs it)
      c = 0;
      if (n_units != U) ab_user_prefix(ctl, ubefore, order, false, n_user, [&](int u) { return H * qtiles_of(u); });
      n_units = U;
    }
  } else if (n_user > 1 && n_user <= kLptMaxUsersFused) {
    // longest first: rank users by key tiles (ties by index)
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
    ab_user_prefix(ctl, ubefore, order, true, n_user, [&](int u) { return H * qtiles_of(u); });
  }
  // unit (or chunk) i -> work item
  auto decode = [&](int i, WorkItem& w) {
    int lo = 0, hi = n_user - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ubefore[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int u = lpt ? order[lo] : lo;
    const int r = cs[u + 1] - cs[u];
    const int L = off[u + 1] - off[u];
    const int nq = qtiles_of(u), s = splits_of(u, c), n = tiles_of(u);
    const int local = i - ubefore[lo];
    const int h = local / (nq * s), rest = local - h * (nq * s);
    const int qt = rest / s, k = rest - qt * s;
    // chunk k of s: key tiles [k n / s, (k + 1) n / s)
    const int t0 = (int)((int64_t)k * n / s), t1 = (int)((int64_t)(k + 1) * n / s);
    w.user = u;
    w.head = h;
    w.cand_begin = cs[u] + qt * cpt;
    w.n_cand = min(cpt, r - qt * cpt);
    w.kv_begin = off[u] + t0 * kBlockN;
    w.kv_len = min(L, t1 * kBlockN) - t0 * kBlockN;
    w.q_row = -1;
    w.n_split = s;
    w.unit = s > 1 ? i - k : -1;      // the chunk index (and CTA) of the unit's first chunk
    w.unit_first = k;
  };
  trace_pro(p, 3);
  WorkItem* mine = p.cta_items + (size_t)b * p.max_cta_items;
  if (n_units <= grid) {
    if (tid == 0) {
      int count = 0;
      if (b < n_units) {
        decode(b, ctl->items[0]);
        count = 1;
      }
      ctl->n_my_items = count;
    }
  } else {
    const int full = n_units / grid, rem = n_units - full * grid;
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
    ctl->mode = kModeIndep;
    ctl->total_keys = off[n_user];
    ctl->ab_chunk_tiles = c;
  }
  trace_pro(p, 7);
  return n_units;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
ikbo_attn_ab_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap qmap1,
                    const __grid_constant__ CUtensorMap kmap_tmpl,
                    const __grid_constant__ CUtensorMap vmap_tmpl) {
  using C = AbConfig<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* data = smem_raw;
  TcCtrl* ctl = reinterpret_cast<TcCtrl*>(smem_raw + kDataBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool layout_ok = (ptx::smem_addr(smem_raw) & 1023u) == 0;
  trace_pro(p, 0);

  if (threadIdx.x == 0) {
    for (int g = 0; g < kAbGroups; ++g) {
      ptx::mbar_init(ptx::smem_addr(&ctl->q_full[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->q_empty[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[g]), 4);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_half[g]), 4);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_free[g]), 4);
      ptx::mbar_init(ptx::smem_addr(&ctl->pv_done[g]), 1);   // a PV of warpgroup g complete (one per tile)
    }
    for (int i = 0; i < kMaxSlots; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_empty[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    // the two softmax warpgroups' rendezvous in the epilogue: one arrival per warp
    ptx::mbar_init(ptx::smem_addr(&ctl->pair_go), 4 * kAbGroups);
    ctl->abort_flag = 0;
    ctl->flags = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 2 && lane == 0) {
    ptx::prefetch_tensormap(&qmap);
    ptx::prefetch_tensormap(&kmap_tmpl);
    ptx::prefetch_tensormap(&vmap_tmpl);
  }
  if (p.fused && layout_ok) plan_load(p, data);
  __syncthreads();
  trace_pro(p, 1);
  int n_units = 0;
  if (!layout_ok || !p.fused) {
    // this kernel plans in-kernel only; the host never launches it otherwise
    if (threadIdx.x == 0) {
      ctl->mode = kModeSkip;
      ctl->n_my_items = 0;
      ctl->sorted = 1;
      atomicOr(p.err_word, kErrLayout);
    }
  } else {
    // no L2 prefetch: the first tiles' loads would queue behind it
    const int flags = plan_group(p, ctl, data, D, false);
    if (flags >= 0) {
      trace_pro(p, 6);
      n_units = plan_ab(p, ctl, data);
      if (threadIdx.x == 0) ctl->sorted = (flags & kPlanUnsorted) ? 0 : 1;
    }
    // the planning scratch is overwritten by TMA (async proxy) from here on
    ptx::fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) ctl->bmaps_ready = 0;   // the planning's scan words are free now
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  trace_pro(p, 8);
  if (threadIdx.x == 0) trace(p, 0, kTrCtaStart);

  const uint32_t tmem = ctl->tmem_base;
  const int mode = ctl->mode;
  const int n_my = ctl->n_my_items;
  const bool sorted = ctl->sorted != 0;
  const int NS = C::kSlots;
  const int Lq = p.Lq;
  uint8_t* q_smem = data;
  uint8_t* p_smem = data + C::kQBufs * C::kQBytes;          // P of warpgroup g at g * kPBytes
  uint8_t* kv_smem = p_smem + kAbGroups * C::kPBytes;
  const int32_t* perm = p.perm_ws;
  const Waiter W{&ctl->abort_flag, p.err_word, p.timeout_ns};
  auto item_at = [&](int k) -> WorkItem {
    return k < kCtlItems ? ctl->items[k] : p.cta_items[(size_t)blockIdx.x * p.max_cta_items + k];
  };
  auto ntiles = [](const WorkItem& w) { return ceil_div(w.kv_len, kBlockN); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (mode != kModeSkip) {
      bool tail_ready = false;
      // K/V maps with an open row count; a tile reaching past row T goes
      // through a copy with the row count set to T (zero fill past the end)
      auto kv_map = [&](bool is_v, int32_t row) -> const void* {
        const int T = ctl->total_keys;
        if (row + kBlockN <= T) return is_v ? (const void*)&vmap_tmpl : (const void*)&kmap_tmpl;
        CUtensorMap* tail_k = p.map_slots + (size_t)p.map_stride * blockIdx.x;
        CUtensorMap* tail_v = tail_k + 1;
        if (!tail_ready) {
          if (lane == 0) {
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
          }
          __syncwarp();
          ptx::tensormap_acquire(tail_k);
          ptx::tensormap_acquire(tail_v);
          tail_ready = true;
        }
        return is_v ? (const void*)tail_v : (const void*)tail_k;
      };
      uint32_t kv_it = 0, q_it = 0;
      // A user's partial last V tile goes through the item's copy of the V
      // map bounded at the user's end row (the TMA fills the other users'
      // rows with zeros), written by warp 2 after planning.
      bool bm_ready = false;
      int cur_item = 0;
      auto v_map_for = [&](int32_t row, int32_t end) -> const void* {
        if (row + kBlockN <= end) return kv_map(true, row);
        if (!bm_ready) {
          bool got = true;
          if (lane == 0) got = wait_bounded_maps(p, ctl);
          if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) return nullptr;
          bm_ready = true;
        }
        CUtensorMap* m = p.map_slots + (size_t)p.map_stride * blockIdx.x + 2 + cur_item;
        ptx::tensormap_acquire(m);
        ptx::prefetch_tensormap(m);
        return m;
      };
      // the next ring load; the item's keys end at row `end`
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
      auto load_q = [&](const WorkItem& w) -> bool {
        const uint32_t qb = q_it % C::kQBufs;
        if (!W.conv_wait(ptx::smem_addr(&ctl->q_empty[qb]), ((q_it / C::kQBufs) & 1u) ^ 1u)) return false;
        ++q_it;
        if (p.debug_flags & 1) return true;    // test hook: never arm the Q barrier
        const uint32_t qbar = ptx::smem_addr(&ctl->q_full[qb]);
        const uint32_t qdst = ptx::smem_addr(q_smem + qb * C::kQBytes);
        if (sorted) {
          const int nb = p.qbox;
          const int nbox = ceil_div(w.n_cand, nb);
          ptx::mbar_arrive_expect_tx_warp(qbar, uint32_t(nbox * nb * Lq * 128 * C::kCB));
          for (int cb = 0; cb < C::kCB; ++cb)
            for (int bx = 0; bx < nbox; ++bx)
              ptx::tma_load_4d_warp(qdst + cb * kTileM * 128 + bx * nb * Lq * 128, &qmap, qbar, cb * 64, 0,
                                    w.head, w.cand_begin + bx * nb);
        } else {
          ptx::mbar_arrive_expect_tx_warp(qbar, uint32_t(w.n_cand * Lq * 128 * C::kCB));
          for (int i = 0; i < w.n_cand; ++i) {
            const int32_t c = perm[w.cand_begin + i];
            for (int cb = 0; cb < C::kCB; ++cb)
              ptx::tma_load_4d_warp(qdst + cb * kTileM * 128 + i * Lq * 128, &qmap1, qbar, cb * 64, 0, w.head, c);
          }
        }
        return true;
      };
      bool ok = true;
      for (int k = 0; k < n_my && ok; ++k) {
        const WorkItem w = item_at(k);
        const int n = ntiles(w);
        if (lane == 0) trace(p, k, kTrProdItem);
        // the MMA warp's order: K0, K1, then per pair of tiles (2i, 2i + 1)
        // K_(2i+2), K_(2i+3), V_(2i), V_(2i+1)
        const int32_t end = w.kv_begin + w.kv_len;
        cur_item = k;
        ok = load_q(w) && ring(false, w.head, w.kv_begin, end) &&
             (n < 2 || ring(false, w.head, w.kv_begin + kBlockN, end));
        for (int j0 = 0; j0 < n && ok; j0 += kAbGroups) {
          for (int j = j0; j < j0 + kAbGroups && ok; ++j)
            if (j + kAbGroups < n) ok = ring(false, w.head, w.kv_begin + (j + kAbGroups) * kBlockN, end);
          for (int j = j0; j < j0 + kAbGroups && j < n && ok; ++j)
            ok = ring(true, w.head, w.kv_begin + j * kBlockN, end);
        }
        if (lane == 0) trace(p, k, kTrProdIssued);
      }
      // Drain: every armed barrier phase must complete before the CTA exits.
      if (lane == 0) {
        for (uint32_t s = 0; s < (uint32_t)NS && s < kv_it; ++s) {
          const uint32_t uses = (kv_it - s + NS - 1) / NS;
          W.drain(ptx::smem_addr(&ctl->kv_full[s]), (uses - 1) & 1u);
        }
        if (!(p.debug_flags & 1))
          for (uint32_t qb = 0; qb < (uint32_t)C::kQBufs && qb < q_it; ++qb) {
            const uint32_t uses = (q_it - qb + C::kQBufs - 1) / C::kQBufs;
            W.drain(ptx::smem_addr(&ctl->q_full[qb]), (uses - 1) & 1u);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (mode != kModeSkip) {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kTileM, kBlockN, 0);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kTileM, D, 1);
      uint32_t kv_it = 0, q_it = 0;
      uint32_t pn[kAbGroups] = {0, 0}, sf[kAbGroups] = {0, 0};
      // the next ring entry, in the producer's order
      auto next_slot = [&](uint32_t& slot) -> bool {
        slot = kv_it % NS;
        if (!W.conv_wait(ptx::smem_addr(&ctl->kv_full[slot]), (kv_it / NS) & 1u)) return false;
        ptx::tc_fence_after();
        return true;
      };
      auto issue_s = [&](int g, uint32_t q_base, uint32_t kslot) {
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
      // O_g += P_g V over keys [64 h, 64 h + 64), P (K-major, 128-byte
      // swizzle, keys 64 h .. 64 h + 63 in its column block h) from shared
      // memory, only the 16-key groups below `groups`
      auto issue_pv_half = [&](int g, uint32_t vslot, int h, bool acc) {
        const uint32_t v_base = ptx::smem_addr(kv_smem + vslot * C::kKVBytes);
        const uint32_t p_base = ptx::smem_addr(p_smem + g * C::kPBytes);
#pragma unroll
        for (int q = 0; q < kBlockN / 32; ++q) {
          const int kk = h * (kBlockN / 32) + q;
          const uint64_t adesc = ptx::smem_desc_sw128(p_base + h * kTileM * 128 + q * 32, 16, 1024);
          const uint64_t bdesc = ptx::smem_desc_sw128(v_base + kk * 16 * 128, kBlockN * 128, 1024);
          ptx::mma_ss_warp(tmem + C::kOCol(g), adesc, bdesc, kIdescPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      auto p_ready = [&](int g, int h) -> bool {
        if (!W.conv_wait(ptx::smem_addr(h == 0 ? &ctl->p_half[g] : &ctl->p_full[g]), pn[g] & 1u)) return false;
        if (h == 1) ++pn[g];
        ptx::tc_fence_after();
        return true;
      };
      bool ok = true;
      for (int k = 0; k < n_my && ok; ++k) {
        const WorkItem w = item_at(k);
        const int n = ntiles(w);
        const uint32_t qb = q_it % C::kQBufs;
        if (!W.conv_wait(ptx::smem_addr(&ctl->q_full[qb]), (q_it / C::kQBufs) & 1u)) break;
        ptx::tc_fence_after();
        if (lane == 0) trace(p, k, kTrMmaQ);
        const uint32_t q_base = ptx::smem_addr(q_smem + qb * C::kQBytes);
        // S_A(0) and S_B(0)
        for (int g = 0; g < kAbGroups && g < n && ok; ++g) {
          uint32_t slot;
          if (!next_slot(slot)) {
            ok = false;
            break;
          }
          issue_s(g, q_base, slot);
          if (g == n - 1) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[qb]));
          ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[slot]));
          ++kv_it;
        }
        if (lane == 0) trace(p, k, kTrMmaFirstS);
        // Per pair of tiles (2i, 2i + 1): first the next S of both warpgroups
        // (each as soon as that warpgroup has its current scores in
        // registers), then both P.V, so that neither warpgroup waits for the
        // other's P.
        for (int j0 = 0; j0 < n && ok; j0 += kAbGroups) {
          for (int j = j0; j < j0 + kAbGroups && ok; ++j) {
            if (j + kAbGroups >= n) continue;
            const int g = j & 1;
            // S_g of tile j + 2 into the buffer warpgroup g has read tile j from
            // (P goes to shared memory, not to this buffer)
            if (!W.conv_wait(ptx::smem_addr(&ctl->s_free[g]), sf[g] & 1u)) {
              ok = false;
              break;
            }
            ++sf[g];
            ptx::tc_fence_after();
            uint32_t kslot;
            if (!next_slot(kslot)) {
              ok = false;
              break;
            }
            issue_s(g, q_base, kslot);
            if (lane == 0 && j < 8) trace_tile(p, k, 2, 2 * j + 1);
            if (j + kAbGroups == n - 1) ptx::mma_commit_warp(ptx::smem_addr(&ctl->q_empty[qb]));
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[kslot]));
            ++kv_it;
          }
          for (int j = j0; j < j0 + kAbGroups && j < n && ok; ++j) {
            const int g = j & 1;
            uint32_t vslot;
            if (!next_slot(vslot)) {
              ok = false;
              break;
            }
            // O_g += P_g V_j, each half of P once the softmax has written it
            if (!p_ready(g, 0)) {
              ok = false;
              break;
            }
            issue_pv_half(g, vslot, 0, j >= kAbGroups);
            if (!p_ready(g, 1)) {
              ok = false;
              break;
            }
            issue_pv_half(g, vslot, 1, true);
            if (lane == 0 && j < 8) trace_tile(p, k, 2, 2 * j);
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->kv_empty[vslot]));
            ptx::mma_commit_warp(ptx::smem_addr(&ctl->pv_done[g]));
            ++kv_it;
          }
        }
        if (lane == 0) trace(p, k, kTrMmaLastPV);
        ++q_it;
      }
      // All issued MMAs must finish before tensor memory is released.
      ptx::mma_commit_warp(ptx::smem_addr(&ctl->drain));
      if (lane == 0) W.drain(ptx::smem_addr(&ctl->drain), 0);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    if (warp == 2 && mode != kModeSkip) write_bounded_maps(p, ctl, &vmap_tmpl, n_my, item_at);
  } else if (mode != kModeSkip) {
    // ------------------------------------------- softmax / correction / epilogue
    const int g = (warp - kSoftmaxWarp0) >> 2;               // warpgroup: even (0) or odd (1) key tiles
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;                      // TMEM lane == tile row
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    const uint32_t scol = tmem + lane_off + C::kSCol(g);
    const float sl2 = p.scale_log2;
    uint32_t tn = 0;                                          // S tiles (and PVs) of this warpgroup so far
    uint32_t pvw = 0;                                         // this warpgroup's PVs waited for
    uint32_t ep = 0;                                          // rendezvous phases so far
    uint8_t* const pbuf = p_smem + g * C::kPBytes;           // this warpgroup's P
    // PV of this warpgroup's tile `pvw` complete (every phase waited in order)
    auto pv_wait = [&]() -> bool {
      if (!W.warp_wait(ptx::smem_addr(&ctl->pv_done[g]), pvw & 1u)) return false;
      ++pvw;
      ptx::tc_fence_after();
      return true;
    };
    // Both warpgroups meet here (every warp arrives, then waits, bounded):
    // what each wrote to shared memory before is visible to the other after.
    // A barrier instruction would not do: a warp that gave up on a wait would
    // leave the others blocked in it.
    const uint32_t epi_bar = ptx::smem_addr(&ctl->pair_go);
    auto rendezvous = [&]() -> bool {
      ptx::mbar_arrive_warp(epi_bar);
      const bool ok = W.warp_wait(epi_bar, ep & 1u);
      ++ep;
      return ok;
    };
    for (int k = 0; k < n_my; ++k) {
      const WorkItem w = item_at(k);
      const int n = ntiles(w);
      const int ng = (n + 1 - g) >> 1;                        // key tiles of this warpgroup
      const bool has_b = n > 1;
      const int rows = w.n_cand * Lq;
      // Rows past the tile's queries hold stale shared memory; their results
      // are never stored, and they are left out of every decision below.
      const bool live = row < rows;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < ng; ++i, ++tn) {
        const int j = 2 * i + g;
        if (!W.warp_wait(ptx::smem_addr(&ctl->s_full[g]), tn & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (i == 0 && row == 0 && g == 0) trace(p, k, kTrSmS0);
        const bool tr_t = row == 0 && j < 4;
        if (tr_t) trace_tile(p, k, 1, 4 * j);
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(scol + c * 32, r[c]);
        ptx::tmem_ld_wait();
        // the scores are in registers: the MMA warp may compute S of tile j + 2
        // into this buffer now
        if (j + kAbGroups < n) {
          ptx::tc_fence_before();
          ptx::mbar_arrive_warp(ptx::smem_addr(&ctl->s_free[g]));
        }
#define IKBO_R(e) __uint_as_float(r[(e) >> 5][(e) & 31])
        // Scores enter the exponent as fma(s, sc, -m): raw scores with
        // sc = scale on full tiles for scale > 0, else scaled here with the
        // keys past the user's sequence at -inf (sc = 1).
        const int valid = min(kBlockN, w.kv_len - j * kBlockN);
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
        if (tr_t) trace_tile(p, k, 1, 4 * j + 1);
        // the running maximum moves only when the tile's exceeds it by more
        // than kLazyRescale, and always on the warpgroup's first tile
        const float m_new = (i == 0 || mx > m + kLazyRescale) ? mx : m;
        const float alpha = fast_exp2(m - m_new);
        // the warpgroup's previous PV must be complete before O_g is rescaled
        // and before P_g is overwritten (it reads both)
        if (i > 0 && !pv_wait()) {
          ok = false;
          break;
        }
        if (i > 0 && __any_sync(0xffffffffu, live && m_new != m)) {
          // O_g holds exactly the warpgroup's earlier tiles
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            ptx::tmem_ld16(tmem + lane_off + C::kOCol(g) + c * 16, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            ptx::tmem_st16(tmem + lane_off + C::kOCol(g) + c * 16, o);
          }
        }
        // P = 2^(s sc - m_new) as bf16 pairs into shared memory, in two halves
        // of 64 keys (the MMA warp starts on the first while the second is
        // made).  Row `row` of column block h: 128 bytes, its 16-byte chunk c
        // (keys 64 h + 8 c ..) at chunk c ^ (row % 8): the 128-byte swizzle
        // the MMA's descriptor reads.
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
          uint8_t* prow = pbuf + h * kTileM * 128 + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) =
                make_uint4(r[h][4 * c], r[h][4 * c + 1], r[h][4 * c + 2], r[h][4 * c + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          ptx::mbar_arrive_warp(ptx::smem_addr(h == 0 ? &ctl->p_half[g] : &ctl->p_full[g]));
          if (tr_t) trace_tile(p, k, 1, 4 * j + 2 + h);
        }
#undef IKBO_R
        l = l * alpha + sum;
        m = m_new;
      }
      if (!ok) break;
      // ---- epilogue: the two warpgroups' results of every row merged; each
      // warpgroup finishes half of the output columns
      ctl->ab_ml[g][row] = make_float2(m, l);
      // this warpgroup's last PV; the other's is waited for by its own warps
      // before the rendezvous
      if (ng > 0 && !pv_wait()) break;
      if (!rendezvous()) break;
      ptx::tc_fence_after();
      if (row == 0 && g == 0) trace(p, k, kTrEpiO);
      const float2 mlA = ctl->ab_ml[0][row], mlB = ctl->ab_ml[1][row];
      const float M = has_b ? fmaxf(mlA.x, mlB.x) : mlA.x;
      const float fa = mlA.x > -INFINITY ? fast_exp2(mlA.x - M) : 0.f;
      const float fb = (has_b && mlB.x > -INFINITY) ? fast_exp2(mlB.x - M) : 0.f;
      const float Lsum = fa * mlA.y + fb * mlB.y;
      const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
      const float lse = Lsum > 0.f ? M + fast_log2(Lsum) : -INFINITY;
      const int split = w.n_split;
      const bool owner = split > 1 && w.unit == (int)blockIdx.x;
      const bool partial = split > 1 && !owner;   // a chunk that is not its unit's first
      // Weights of this row's own result (a) and of the other chunks' (as),
      // all divided by their sum: the merge of the chunks of a unit by the
      // log-sum-exp rule, out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
      float wself = 1.f;
      float wpeer[kAbMaxSplit];
#pragma unroll
      for (int s2 = 0; s2 < kAbMaxSplit; ++s2) wpeer[s2] = 0.f;
      if (owner) {
        // wait (bounded) for the flags of the unit's other chunks: lanes 1 ..
        // split - 1 of the first softmax warp, one flag each; then reset them
        if (warp == kSoftmaxWarp0) {
          bool got = true;
          if (lane >= 1 && lane < split) {
            unsigned long long* f = p.ab_flags + blockIdx.x + lane;
            uint64_t t_end = 0;
            unsigned long long v = 0;
            for (uint32_t spin = 0;; ++spin) {
              asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
              if (v == p.ab_marker) break;
              if ((spin & 15u) == 15u) {
                if (*W.abort) {
                  got = false;
                  break;
                }
                const uint64_t now = ptx::globaltimer();
                if (t_end == 0) {
                  t_end = now + p.timeout_ns;
                } else if (now > t_end) {
                  *W.abort = 1;
                  atomicOr(p.err_word, kErrTimeout);
                  got = false;
                  break;
                }
              }
            }
            if (got) *f = 0ull;
          }
          const bool all = __all_sync(0xffffffffu, got);
          if (lane == 0) ctl->flags = all ? 1 : 0;
        }
        if (!rendezvous()) break;
        if (row == 0 && g == 0) trace(p, k, kTrArrived);
        if (ctl->flags != 1) break;
        float lp[kAbMaxSplit];
        float Mx = lse;
#pragma unroll
        for (int s2 = 1; s2 < kAbMaxSplit; ++s2) {
          lp[s2] = (live && s2 < split) ? __ldcg(p.ab_partial_lse + (size_t)(blockIdx.x + s2) * kTileM + row)
                                        : -INFINITY;
          Mx = fmaxf(Mx, lp[s2]);
        }
        float den = lse > -INFINITY ? fast_exp2(lse - Mx) : 0.f;
        wself = den;
#pragma unroll
        for (int s2 = 1; s2 < kAbMaxSplit; ++s2) {
          wpeer[s2] = lp[s2] > -INFINITY ? fast_exp2(lp[s2] - Mx) : 0.f;
          den += wpeer[s2];
        }
        const float id = den > 0.f ? 1.f / den : 0.f;
        wself *= id;
#pragma unroll
        for (int s2 = 1; s2 < kAbMaxSplit; ++s2) wpeer[s2] *= id;
      }
      const float2 wa = make_float2(fa * inv * wself, fa * inv * wself);
      const float2 wb = make_float2(fb * inv * wself, fb * inv * wself);
      const int col0 = g * C::kHalf;
      const uint32_t oa = tmem + lane_off + C::kOCol(0) + col0;
      const uint32_t ob = tmem + lane_off + C::kOCol(1) + col0;
      // the output row (unless this chunk only hands its result on)
      const int ci = live ? row / Lq : 0;
      const int tq = live ? row - ci * Lq : 0;
      const int32_t gpos = w.cand_begin + ci;
      const int64_t cidx = (live && !partial) ? (sorted ? gpos : perm[gpos]) : 0;
      uint16_t* dst = p.out + (((cidx * p.H + w.head) * (int64_t)Lq + tq) * D) + col0;
      const size_t slot = blockIdx.x;
      float4* po = p.ab_partial_o + slot * (D / 4) * kTileM;
      // 32 columns at a time: O of both warpgroups from tensor memory, merged
      // (one chunk in registers at a time)
#pragma unroll 1
      for (int c = 0; c < C::kHalf / 32; ++c) {
        // (O_B is read even when warpgroup B had no tile, and then not used:
        // a load under a condition costs the kernel its registers)
        uint32_t va[32], vb[32];
        ptx::tmem_ld32(oa + c * 32, va);
        ptx::tmem_ld32(ob + c * 32, vb);
        ptx::tmem_ld_wait();
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float2 y = fmul2(make_float2(__uint_as_float(va[e]), __uint_as_float(va[e + 1])), wa);
          if (has_b) y = ffma2(make_float2(__uint_as_float(vb[e]), __uint_as_float(vb[e + 1])), wb, y);
          x[e] = y.x;
          x[e + 1] = y.y;
        }
        if (!live) continue;
        const int c4base = (col0 + c * 32) / 4;
        if (partial) {
          // O / l of this chunk's rows to global memory (16-byte column groups, row-minor)
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            po[(size_t)(c4base + q4) * kTileM + row] = make_float4(x[4 * q4], x[4 * q4 + 1], x[4 * q4 + 2], x[4 * q4 + 3]);
          continue;
        }
        if (owner) {
#pragma unroll
          for (int s2 = 1; s2 < kAbMaxSplit; ++s2) {
            if (s2 >= split) break;
            const float4* pp4 = p.ab_partial_o + (size_t)(blockIdx.x + s2) * (D / 4) * kTileM;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 y = __ldcg(pp4 + (size_t)(c4base + q4) * kTileM + row);
              x[4 * q4] += wpeer[s2] * y.x;
              x[4 * q4 + 1] += wpeer[s2] * y.y;
              x[4 * q4 + 2] += wpeer[s2] * y.z;
              x[4 * q4 + 3] += wpeer[s2] * y.w;
            }
          }
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        store_bf16x32(dst + c * 32, w);
      }
      if (partial && live && g == 0) p.ab_partial_lse[slot * kTileM + row] = lse;
      // The next item's first PVs overwrite O_A and O_B: both warpgroups are
      // done reading before either hands over that item's first P.  A chunk
      // that hands its result on raises its flag once every row is written.
      ptx::tc_fence_before();
      if (partial) __threadfence();
      if (!rendezvous()) break;
      if (partial && warp == kSoftmaxWarp0 && lane == 0)
        asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.ab_flags + slot), "l"(p.ab_marker) : "memory");
      if (row == 0 && g == 0) trace(p, k, owner ? kTrMerged : kTrEpiStored);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace(p, 0, kTrCtaEnd);
  trace_pro(p, 10);
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace ikbo
