// IKBO linear compression on the 5th-generation tensor cores (sm_103a).
//
// What it computes ("In-Kernel Broadcast Optimization: Co-Designing Kernels
// for RecSys Inference", §2): linear compression of embeddings projects each
// candidate's K input embeddings X[b] (K x N) with a learned W (M x K),
// out[b] = W @ X[b].  The K embeddings are the candidate's user's block
// followed by its own, so with W = [W_user | W_cand]
//
//     out[b] = W_user @ X_user[u(b)] + W_cand @ X_cand[b],   u(b) = cand_to_user[b]
//
// (§2.1: the broadcast pushed past the matrix product; the user term is
// computed once per user, at the user batch size).  Two stages, one kernel:
//   stage 0  Y[u] = W_user @ X_user[u] for every user, accumulated in fp32
//            and kept in bf16 (the term is read once per candidate and row
//            tile, 128 x N values each time: bf16 halves those reads);
//   stage 1  out[b] = W_cand @ X_cand[b] + Y[u(b)]: the broadcast add is fused
//            into the epilogue (§2.3), which finds Y through cand_to_user, so
//            no broadcast tensor is ever written.
// A user -> vendor -> item hierarchy (§5: two nested broadcasts) adds a level
// in the middle: Y_vendor[v] = W_vendor @ X_vendor[v] + Y_user[vendor_to_user[v]]
// (in bf16), then out[i] = W_item @ X_item[i] + Y_vendor[item_to_vendor[i]].
// A launch is one level: its product, plus, in the epilogue, the bf16 term of
// the level above found through one map (or, when the middle level has no
// block, through both maps), summed in fp32 and stored in bf16 (the output,
// or the term of the level below).
// Each K block arrives zero-padded to a multiple of 8 (§2.2), so every row is
// 16-byte aligned for the TMA.
//
// Work unit: (batch index, 128-row tile of M).  Persistent CTAs, warp roles
// (256 threads):
//   warp 0     TMA producer: per 64-wide step of K, the W tile (128 x 64,
//              K-major) and the X tile (64 x N, N contiguous) into a ring;
//   warp 1     MMA warp, converged, one elected lane issuing: D = W X in
//              tensor memory (M = 128, N = the full width, K = 16 per MMA),
//              two accumulators so that the epilogue of one unit overlaps the
//              MMAs of the next;
//   warps 4-7  epilogue: TMEM lane r = row r of the tile; 32 columns at a time,
//              + Y of the level above, rounded to bf16 into a shared-memory
//              staging box (each warp its 32 rows x 64 columns, two boxes in
//              turn), which the warp's TMA store writes out: whole 128-byte
//              lines, where one row per thread would write 16 bytes to each
//              of 32 rows 512 bytes apart.
// Each level is launched as a programmatic dependent of the one above; only
// its epilogue waits for the Y it adds, so its loads and MMAs overlap the
// level above.
//
// Clusters (M of at most 8 row tiles): the CTAs of a cluster take the row
// tiles of one batch entry at a time, CTA r tile r.  A cluster runs on one
// die, so the X tile that all its CTAs load comes from DRAM once and from
// that die's L2 for the others.
//
// Two forms:
//   kPair = false  every CTA computes its 128 rows alone (M = 128 MMAs); the
//                  CTAs touch nothing of one another, each loads its own W
//                  and the whole X tile into its own ring;
//   kPair = true   CTAs 2i and 2i + 1 of the cluster compute 256 rows
//                  together with M = 256 MMAs over both tensor cores
//                  (cta_group::2).  Each CTA loads its own 128 rows of W and
//                  HALF of the X tile's columns (the even CTA the first N/2,
//                  the odd one the rest): per K step a CTA takes in 32 KB
//                  instead of 48 KB at N = 256, and its tensor core reads
//                  8 KB of shared memory per MMA instead of 12.  The even CTA
//                  issues every MMA; both CTAs' loads complete on the even
//                  CTA's ring barrier; each MMA commit arrives on the ring,
//                  accumulator and drain barriers of both CTAs; the odd CTA's
//                  epilogue hands its accumulator back to the even CTA's
//                  barrier.  Each CTA's epilogue reads its own 128 rows from
//                  its own tensor memory.
// Teardown: every byte that reaches a CTA is counted on a ring barrier that a
// producer drains; with CTA pairs no CTA leaves before its cluster has.
// Every wait is bounded, as in the attention kernels.
#pragma once

#include "ikbo_attn_tc.cuh"

namespace ikbo {

constexpr int kLceThreads = 256;
constexpr int kLceEpiWarp0 = 4;
constexpr int kLceKStep = 64;                  // K per ring stage (one 128-byte swizzle atom of bf16)
constexpr int kLceSmemBytes = 232448;          // the per-CTA maximum
constexpr int kLceCtrlBytes = 1024;
constexpr int kLceEpiBoxBytes = 32 * 64 * 2;   // one epilogue warp's store box: 32 rows x 64 bf16
constexpr int kLceEpiBytes = 4 * 2 * kLceEpiBoxBytes;   // 4 warps x 2 boxes
constexpr int kLceMaxStages = 8;

struct LceParams {
  const uint16_t* W;          // bf16 [M, K] of this level's block
  const int32_t* map;         // add: batch entry -> entry of the level above
  const int32_t* map2;        // add, or null: entry of the level above -> the one above that
  const uint16_t* Y;          // add: bf16 [rows, M, N] terms of the level(s) above
  uint16_t* out;              // bf16 [n_batch, M, N]: the output, or the term of the level below
  int64_t n_batch;            // entries of this level (users, vendors, candidates or items)
  int64_t n_map;              // map values must lie in [0, n_map)
  int64_t n_map2;             // map2 values must lie in [0, n_map2)
  int32_t M, K, N;
  int32_t add;                // 1: add a row of Y (after the grid above has completed)
  int32_t y_via_map2;         // add with map2: 1 = Y row map2[map[b]]; 0 = Y row map[b], map2 only checked
  int32_t has_dependent;      // 1: the level below is this grid's programmatic dependent
  int32_t cluster_n;          // CTAs per cluster: the row tiles of M (<= 8), or 1 (co-scheduling only)
  int* err_word;
  uint64_t timeout_ns;
};

template <int NB, bool kPair = false>
struct LceConfig {
  static constexpr int N = NB * 64;
  static constexpr int kXBlocks = kPair ? NB / 2 : NB;  // 64-column blocks of X this CTA loads
  static constexpr int kABytes = kTileM * 128;          // 128 rows x 64 bf16
  static constexpr int kBBytes = kXBlocks * kLceKStep * 128;  // blocks of 64 rows x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages0 = (kLceSmemBytes - kLceCtrlBytes - kLceEpiBytes) / kStageBytes;
  static constexpr int kStages = kStages0 < kLceMaxStages ? kStages0 : kLceMaxStages;
  static constexpr int kDataBytes = kStages * kStageBytes;   // the ring, then the epilogue boxes
  static_assert(kStages >= 2, "ring");
  static_assert(kDataBytes % 1024 == 0, "epilogue boxes 1 KB aligned (128-byte swizzle)");
  static_assert(kDataBytes + kLceEpiBytes + kLceCtrlBytes <= kLceSmemBytes, "shared memory");
  static_assert(2 * N <= 512, "two accumulators in tensor memory");
  static_assert(!kPair || NB % 2 == 0, "CTA pairs split X into halves of whole 64-column blocks");
};

struct LceCtrl {
  uint64_t full[kLceMaxStages], empty[kLceMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(LceCtrl) <= kLceCtrlBytes, "control block");

template <int NB, bool kPair>
__global__ void __launch_bounds__(kLceThreads, 1)
ikbo_lce_kernel(const __grid_constant__ LceParams p, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap omap) {
  using C = LceConfig<NB, kPair>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* data = smem_raw;
  uint8_t* epi_smem = smem_raw + C::kDataBytes;
  LceCtrl* ctl = reinterpret_cast<LceCtrl*>(smem_raw + C::kDataBytes + kLceEpiBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the level below may start at once (it waits for this level's Y only in
  // its epilogue)
  if (p.has_dependent) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const bool layout_ok = (ptx::smem_addr(smem_raw) & 1023u) == 0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->acc_full[i]), 1);
      // the 4 epilogue warps (with CTA pairs, the even CTA's barrier also
      // takes the odd CTA's 4)
      ptx::mbar_init(ptx::smem_addr(&ctl->acc_empty[i]), kPair ? 8 : 4);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
    if (!layout_ok) atomicOr(p.err_word, kErrLayout);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_addr(&ctl->tmem_base), 512);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), 512);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 2 && lane == 0) {
    ptx::prefetch_tensormap(&wmap);
    ptx::prefetch_tensormap(&xmap);
    ptx::prefetch_tensormap(&omap);
  }
  ptx::tc_fence_before();
  // with CTA pairs, the peer's barriers are initialised before any MMA
  // commit or TMA byte reaches them
  if constexpr (kPair) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const Waiter W{&ctl->abort_flag, p.err_word, p.timeout_ns};
  const int mt_count = (p.M + kTileM - 1) / kTileM;
  const int ksteps = (p.K + kLceKStep - 1) / kLceKStep;
  // units: with clusters, the batch entries, one per cluster at a time, row
  // tile = rank; without, (batch entry, row tile) pairs
  const int cn = p.cluster_n;
  const int rank = cn > 1 ? int(ptx::cluster_ctarank()) : 0;
  // CTA pairs: the even CTA (the "leader") issues the MMAs; barrier
  // addresses in both CTAs of the pair
  const bool leader = !kPair || (rank & 1) == 0;
  const uint32_t pair_lead = uint32_t(rank & ~1), pair_odd = uint32_t(rank | 1);
  auto lead_bar = [&](uint64_t* b) { return ptx::map_to_cta(ptx::smem_addr(b), pair_lead); };
  auto odd_bar = [&](uint64_t* b) { return ptx::map_to_cta(ptx::smem_addr(b), pair_odd); };
  const int64_t first = cn > 1 ? blockIdx.x / cn : blockIdx.x;
  const int64_t stride = cn > 1 ? gridDim.x / cn : gridDim.x;
  const int64_t n_units = cn > 1 ? p.n_batch : p.n_batch * mt_count;
  auto unit_bm = [&](int64_t unit, int& b, int& mt) {
    if (cn > 1) {
      b = int(unit);
      mt = rank;
    } else {
      b = int(unit / mt_count);
      mt = int(unit % mt_count);
    }
  };

  if (layout_ok && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t unit = first; unit < n_units && ok; unit += stride) {
        int b, mt;
        unit_bm(unit, b, mt);
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const uint32_t slot = it % C::kStages;
          if (!W.wait(ptx::smem_addr(&ctl->empty[slot]), ((it / C::kStages) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t dst = ptx::smem_addr(data + slot * C::kStageBytes);
          if constexpr (kPair) {
            // both CTAs' bytes complete on the even CTA's barrier, which the
            // even CTA's producer arms for both
            const uint32_t bar = lead_bar(&ctl->full[slot]);
            if (leader) ptx::mbar_arrive_expect_tx(ptx::smem_addr(&ctl->full[slot]), 2 * C::kStageBytes);
            ptx::tma_load_2d_pair(dst, &wmap, bar, ks * kLceKStep, mt * kTileM);
            const int c0 = (rank & 1) * C::kXBlocks;   // this CTA's half of the columns
#pragma unroll
            for (int c = 0; c < C::kXBlocks; ++c)
              ptx::tma_load_3d_pair(dst + C::kABytes + c * kLceKStep * 128, &xmap, bar, (c0 + c) * 64,
                                    ks * kLceKStep, b);
          } else {
            const uint32_t bar = ptx::smem_addr(&ctl->full[slot]);
            ptx::mbar_arrive_expect_tx(bar, C::kStageBytes);
            // W[mt*128 .. +128, k .. k+64] (rows past M and columns past K read as zeros)
            ptx::tma_load_2d(dst, &wmap, bar, ks * kLceKStep, mt * kTileM);
            // X[b, k .. k+64, 64 c .. 64 c + 64] for each 64-column block c
#pragma unroll
            for (int c = 0; c < NB; ++c)
              ptx::tma_load_3d(dst + C::kABytes + c * kLceKStep * 128, &xmap, bar, c * 64, ks * kLceKStep, b);
          }
        }
      }
      // every armed phase must complete before the CTA exits (with CTA
      // pairs the even CTA's barriers count both CTAs' bytes; the odd CTA
      // stays until the cluster's closing barrier)
      if (leader)
        for (uint32_t s = 0; s < (uint32_t)C::kStages && s < it; ++s) {
          const uint32_t uses = (it - s + C::kStages - 1) / C::kStages;
          W.drain(ptx::smem_addr(&ctl->full[s]), (uses - 1) & 1u);
        }
    }
    __syncwarp();
  } else if (layout_ok && warp == 1 && leader) {
    // -------------------------------------------------------------- MMA warp
    // converged; the elected lane issues every MMA and commit
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kPair ? 2 * kTileM : kTileM, C::N, 1);
    // commit to this CTA's barrier and, with CTA pairs, to the odd CTA's too
    auto commit = [&](uint64_t* b) {
      if constexpr (kPair) {
        ptx::mma_commit_pair_warp(ptx::smem_addr(b));
        ptx::mma_commit_pair_warp(odd_bar(b));
      } else {
        ptx::mma_commit_warp(ptx::smem_addr(b));
      }
    };
    uint32_t it = 0, ui = 0;
    bool ok = true;
    for (int64_t unit = first; unit < n_units && ok; unit += stride, ++ui) {
      const uint32_t buf = ui & 1u;
      // the epilogue has read this accumulator's previous unit
      if (!W.conv_wait(ptx::smem_addr(&ctl->acc_empty[buf]), ((ui >> 1) & 1u) ^ 1u)) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + buf * C::N;
      for (int ks = 0; ks < ksteps; ++ks, ++it) {
        const uint32_t slot = it % C::kStages;
        if (!W.conv_wait(ptx::smem_addr(&ctl->full[slot]), (it / C::kStages) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_base = ptx::smem_addr(data + slot * C::kStageBytes);
        const uint32_t b_base = a_base + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < kLceKStep / 16; ++kk) {
          // A: K-major, 128-byte swizzle, 32 bytes per K = 16 step
          const uint64_t adesc = ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
          // B: N contiguous (MN-major): 16 K-rows per step, 64-column blocks
          // kLceKStep * 128 bytes apart, 8-row groups 1 KB apart
          const uint64_t bdesc = ptx::smem_desc_sw128(b_base + kk * 16 * 128, kLceKStep * 128, 1024);
          if constexpr (kPair)
            ptx::mma_ss_pair_warp(d_tmem, adesc, bdesc, kIdesc, (ks > 0 || kk > 0) ? 1u : 0u);
          else
            ptx::mma_ss_warp(d_tmem, adesc, bdesc, kIdesc, (ks > 0 || kk > 0) ? 1u : 0u);
        }
        commit(&ctl->empty[slot]);
      }
      if (!ok) break;
      commit(&ctl->acc_full[buf]);
    }
    commit(&ctl->drain);
    if (lane == 0) W.drain(ptx::smem_addr(&ctl->drain), 0);
    __syncwarp();
  } else if (layout_ok && warp >= kLceEpiWarp0) {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                      // TMEM lane == tile row
    const uint32_t lane_off = uint32_t(quarter * 32) << 16;
    // this warp's two store boxes (32 rows x 64 columns, 128-byte swizzle)
    const uint32_t box0 = ptx::smem_addr(epi_smem + quarter * 2 * kLceEpiBoxBytes);
    uint32_t nbox = 0;          // boxes staged so far (the buffer is nbox & 1)
    bool prev_stored = false;   // the box before was stored (its group may still read)
    bool y_ready = !p.add;
    uint32_t ui = 0;
    for (int64_t unit = first; unit < n_units; unit += stride, ++ui) {
      const uint32_t buf = ui & 1u;
      int b, mt;
      unit_bm(unit, b, mt);
      const int m = mt * kTileM + r;
      const bool live = m < p.M;
      int64_t u = 0;
      bool bad = false;
      if (p.add) {
        if (!y_ready) {
          // Y is the level above's output: visible once that grid has completed
          asm volatile("griddepcontrol.wait;" ::: "memory");
          y_ready = true;
        }
        u = p.map[b];
        bad = u < 0 || u >= p.n_map;
        if (!bad && p.map2) {
          const int64_t top = p.map2[u];
          bad = top < 0 || top >= p.n_map2;
          if (p.y_via_map2) u = top;
        }
        if (bad && r == 0) atomicOr(p.err_word, kErrIndex);
      }
      // The term of the level above for this row, in 32-column chunks: the
      // first kYAhead are requested before the accumulator is waited for (they
      // arrive while the unit's MMAs run), then each kYAhead chunks ahead of
      // its use.
      constexpr int kChunks = C::N / 32;
      constexpr int kYAhead = 2;
      const bool add = p.add && live && !bad;
      const uint4* yrow = add ? reinterpret_cast<const uint4*>(p.Y + (u * p.M + m) * p.N) : nullptr;
      uint4 yb[kYAhead + 1][4];
      if (add) {
#pragma unroll
        for (int c = 0; c < kYAhead && c < kChunks; ++c) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) yb[c][q8] = yrow[c * 4 + q8];
        }
      }
      if (!W.warp_wait(ptx::smem_addr(&ctl->acc_full[buf]), (ui >> 1) & 1u)) break;
      ptx::tc_fence_after();
      const uint32_t acc = tmem + lane_off + buf * C::N;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if (add && c + kYAhead < kChunks) {
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) yb[(c + kYAhead) % (kYAhead + 1)][q8] = yrow[(c + kYAhead) * 4 + q8];
        }
        uint32_t o[32];
        ptx::tmem_ld32(acc + c * 32, o);
        ptx::tmem_ld_wait();
        const uint32_t box = box0 + (nbox & 1u) * kLceEpiBoxBytes;
        if ((c & 1) == 0 && !bad && nbox >= 2) {
          // the box's buffer was last stored two boxes ago: that store has
          // read it once at most one group (the box before) is still reading
          if (lane == 0) {
            if (prev_stored) ptx::bulk_wait_read_1(); else ptx::bulk_wait_read_0();
          }
          __syncwarp();
        }
        if (!bad) {
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(o[e]);
          if (add) {
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
              const uint4 t = yb[c % (kYAhead + 1)][q8];
              const uint32_t wv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                x[8 * q8 + 2 * i] += __uint_as_float(wv[i] << 16);
                x[8 * q8 + 2 * i + 1] += __uint_as_float(wv[i] & 0xffff0000u);
              }
            }
          }
          // row `lane` of the box: 16-byte chunk k of the row at k ^ (row % 8)
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            const uint32_t k = uint32_t(((c & 1) * 4 + q8) ^ (lane & 7));
            ptx::st_shared_v4(box + lane * 128 + k * 16, pack_bf16(x[8 * q8], x[8 * q8 + 1]),
                              pack_bf16(x[8 * q8 + 2], x[8 * q8 + 3]), pack_bf16(x[8 * q8 + 4], x[8 * q8 + 5]),
                              pack_bf16(x[8 * q8 + 6], x[8 * q8 + 7]));
          }
          if (c & 1) {
            // the box is complete: the warp's TMA store writes it (rows past M
            // are not written), in a bulk group of its own
            ptx::fence_proxy_async_smem();
            __syncwarp();
            const int y0 = mt * kTileM + quarter * 32;
            const bool store = y0 < p.M;
            if (lane == 0) {
              if (store) ptx::tma_store_3d(&omap, box, (c >> 1) * 64, y0, b);
              ptx::bulk_commit_group();
            }
            prev_stored = store;
            ++nbox;
          }
        }
      }
      // this accumulator may take the next unit's MMAs (with CTA pairs, the
      // even CTA's barrier counts both CTAs' epilogue warps)
      ptx::tc_fence_before();
      if constexpr (kPair) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lead_bar(&ctl->acc_empty[buf]));
      } else {
        ptx::mbar_arrive_warp(ptx::smem_addr(&ctl->acc_empty[buf]));
      }
    }
    // every store has written its box before the CTA leaves
    if (lane == 0) ptx::bulk_wait_all();
    __syncwarp();
  }
  ptx::tc_fence_before();
  if constexpr (kPair) {
    // The even CTA's MMAs read the odd CTA's shared memory and write its
    // tensor memory, and the odd CTA's loads complete on the even CTA's
    // barriers: both leave together, after the even CTA has drained both.
    // The odd CTA also takes the drain commit, once its own roles are done
    // (then the last MMA has completed, or the call has failed), so that it
    // sees the last MMA complete before it frees its tensor memory.
    __syncthreads();
    if (warp == 1 && !leader && layout_ok && lane == 0) W.drain(ptx::smem_addr(&ctl->drain), 0);
    __syncwarp();
    ptx::cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (kPair) ptx::tmem_dealloc_pair(tmem, 512); else ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace ikbo
