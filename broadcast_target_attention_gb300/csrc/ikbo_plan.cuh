// Planning kernel: validate the index tensors, group candidates by user and
// write the work list of the attention kernel.
//
// "In-Kernel Broadcast Optimization", §1.3 item 3: the inference runtime hands
// the kernel a candidate-to-user mapping instead of a materialised broadcast;
// §3.2 assumes the candidates of one user arrive next to each other.  This
// kernel accepts any mapping: sorted input is used as is, otherwise a stable
// counting sort by user produces `perm` (grouped position -> candidate).
//
// Work list order follows two scheduling ideas from the pages:
//  * user-major ("In-Kernel Broadcast Optimization", §3.1, Table 1: the
//    launch grid puts candidates before heads so CTAs sharing a user's K/V
//    run together and hit in L2): the items of one (user, head) are adjacent;
//  * longest first ("Optimizing Jagged Flash Attention with TLX", §2.2,
//    scheduling jagged tiles across SMs: tiles sorted by K/V work, heaviest
//    first): users are emitted by decreasing sequence length, and the
//    persistent attention CTAs take items in that order.
// When the (user, head, query-tile) units are too few to fill the SMs, each
// unit's keys are split into ranges of equal tile count and the partial
// results are merged by log-sum-exp ("Chapter 4: High-performance Kernels",
// §4.6.4, Flash-Decoding).
#pragma once

#include <cuda.h>

#include "ikbo_common.cuh"

namespace ikbo {

// Everything the planner needs besides PlanParams: the output (for users
// with an empty sequence, whose rows are zero) and the K/V tensor-map
// templates whose row count is only known on the device.
struct PlanExtra {
  void* out;
  int32_t Lq;
  int32_t D;
  int32_t patch_maps;   // 1: copy the templates below into *_dst and set their row count to T
  int32_t pad;
  CUtensorMap* kmap_dst;
  CUtensorMap* vmap_dst;
  CUtensorMap kmap_tmpl;
  CUtensorMap vmap_tmpl;
};

constexpr int kPlanThreads = 1024;
constexpr int kLptMaxUsers = 4096;

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Block-wide exclusive scan of int64 values, one value per thread.
// Returns the exclusive prefix; *total receives the block sum.
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t x, int64_t* smem32, int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t v = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) smem32[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int64_t w = lane < nw ? smem32[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem32[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  int64_t warp_prefix = warp == 0 ? 0 : smem32[warp - 1];
  *total = smem32[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_prefix + v - x;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
ikbo_plan_kernel(const __grid_constant__ PlanParams p, const __grid_constant__ PlanExtra x) {
  // The attention kernel may start its prologue now; it waits for this
  // grid's completion (griddepcontrol.wait) before reading the plan.
  asm volatile("griddepcontrol.launch_dependents;");

  __shared__ int s_err;
  __shared__ int s_unsorted;
  // sequence lengths of up to kLptMaxUsers users, for the longest-first order
  __shared__ int32_t s_len[kLptMaxUsers];
  __shared__ int64_t s_scan[32];
  __shared__ int64_t s_sum_units, s_sum_tiles;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;
  const int64_t n_cand = p.n_cand;
  const int64_t n_user = p.n_user;
  // not __restrict__: in a multi-level call it points at item_user, which
  // this kernel writes first (plain loads, no read-only path)
  const int32_t* c2u = p.cand_to_user;
  const int32_t* __restrict__ off = p.user_offsets;

  if (tid == 0) {
    s_err = 0;
    s_unsorted = 0;
  }
  if (p.vendor_to_user) {
    // 0. multi-level call: every item's user through its vendor; an
    // out-of-range vendor becomes -1, which step 1 reports as a bad index
    for (int64_t c = tid; c < n_cand; c += nt) {
      const int32_t vd = p.cand_to_user[c];
      p.item_user[c] = (vd >= 0 && (int64_t)vd < p.n_vendor) ? p.vendor_to_user[vd] : -1;
    }
    c2u = p.item_user;
  }
  __syncthreads();

  // 1. validation -----------------------------------------------------------
  int err = 0;
  if (tid == 0 && off[0] != 0) err |= kErrOffsets;
  for (int64_t u = tid; u < n_user; u += nt)
    if (off[u + 1] < off[u]) err |= kErrOffsets;
  int unsorted = 0;
  for (int64_t c = tid; c < n_cand; c += nt) {
    const int32_t uc = c2u[c];
    if (uc < 0 || (int64_t)uc >= n_user) err |= kErrIndex;
    if (c > 0 && c2u[c - 1] > uc) unsorted = 1;
  }
  if (err) atomicOr(&s_err, err);
  if (unsorted) s_unsorted = 1;
  __syncthreads();
  if (s_err) {
    if (tid == 0) {
      p.header->n_items = 0;
      p.header->error = s_err;
      p.header->work_counter = 0;
      atomicOr(p.err_word, s_err);
    }
    return;
  }
  const bool sorted = !s_unsorted;
  // the sequence lengths, from shared memory in the steps below (up to
  // kLptMaxUsers users; beyond, from the offsets)
  const bool len_smem = n_user <= kLptMaxUsers;
  if (len_smem)
    for (int64_t u = tid; u < n_user; u += nt) s_len[u] = off[u + 1] - off[u];
  auto len_of = [&](int64_t u) -> int32_t { return len_smem ? s_len[u] : off[u + 1] - off[u]; };

  // 2. group candidates by user ---------------------------------------------
  int32_t* cand_start = p.cand_start;
  if (sorted) {
    for (int64_t c = tid; c < n_cand; c += nt) {
      const int32_t uc = c2u[c];
      const int32_t prev = c == 0 ? -1 : c2u[c - 1];
      for (int32_t uu = prev + 1; uu <= uc; ++uu) cand_start[uu] = (int32_t)c;
    }
    for (int64_t uu = (int64_t)c2u[n_cand - 1] + 1 + tid; uu <= n_user; uu += nt)
      cand_start[uu] = (int32_t)n_cand;
  } else {
    int32_t* count = p.scratch;
    for (int64_t u = tid; u < n_user; u += nt) count[u] = 0;
    __syncthreads();
    for (int64_t c = tid; c < n_cand; c += nt) atomicAdd(&count[c2u[c]], 1);
    __syncthreads();
    int64_t carry = 0;
    for (int64_t base = 0; base < n_user; base += nt) {
      const int64_t u = base + tid;
      const int64_t val = u < n_user ? count[u] : 0;
      int64_t tot;
      const int64_t ex = block_exclusive_scan(val, s_scan, &tot);
      if (u < n_user) cand_start[u] = (int32_t)(carry + ex);
      carry += tot;
    }
    if (tid == 0) cand_start[n_user] = (int32_t)n_cand;
    __syncthreads();
    // stable scatter: one warp walks the candidates in order, 32 at a time;
    // lanes that share a user take consecutive slots in lane order.
    if (tid < 32) {
      int32_t* cursor = count;
      for (int64_t u = tid; u < n_user; u += 32) cursor[u] = cand_start[u];
      __syncwarp();
      const unsigned lt = (1u << tid) - 1u;
      for (int64_t base = 0; base < n_cand; base += 32) {
        const int64_t c = base + tid;
        const bool valid = c < n_cand;
        const int32_t uc = valid ? c2u[c] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, uc);
        int32_t pos = 0;
        if (valid) pos = cursor[uc] + __popc(same & lt);
        __syncwarp();
        if (valid && (same & lt) == 0) cursor[uc] += __popc(same);
        if (valid) p.perm[pos] = (int32_t)c;
        __syncwarp();
      }
    }
  }
  __syncthreads();

  // 3. zero rows of candidates whose user has an empty sequence --------------
  {
    const int64_t row_elems = (int64_t)p.H * x.Lq * x.D;   // bf16 elements per candidate
    for (int64_t c = tid; c < n_cand; c += nt) {
      const int32_t uc = c2u[c];
      if (len_of(uc) == 0) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(x.out) + c * row_elems);
        for (int64_t i = 0; i < row_elems / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  // 4. per-user work sizes and the split decision ----------------------------
  const int cpt = p.cands_per_tile;
  const int bn = p.block_n;
  int64_t my_units = 0, my_tiles = 0;
  for (int64_t u = tid; u < n_user; u += nt) {
    const int64_t r = cand_start[u + 1] - cand_start[u];
    const int64_t L = off[u + 1] - off[u];
    if (r > 0 && L > 0) {
      const int64_t nmt = ceil_div64(r, cpt);
      my_units += nmt;
      my_tiles += nmt * ceil_div64(L, bn);
    }
  }
  // block sums (reuse the scan)
  {
    int64_t tot_u, tot_t;
    block_exclusive_scan(my_units, s_scan, &tot_u);
    block_exclusive_scan(my_tiles, s_scan, &tot_t);
    if (tid == 0) {
      s_sum_units = tot_u * p.H;
      s_sum_tiles = tot_t * p.H;
    }
  }
  __syncthreads();
  const int64_t base_units = s_sum_units;
  int64_t split_tiles = 0;
  if (p.allow_split && base_units > 0 && base_units < 2 * (int64_t)p.num_sms) {
    split_tiles = ceil_div64(s_sum_tiles, p.num_sms);
    if (split_tiles < 1) split_tiles = 1;
  }

  // 5. order users (longest sequence first) ---------------------------------
  // scratch[rank] = user.  Users beyond kLptMaxUsers keep their index order.
  int32_t* order = p.scratch;
  if (n_user <= kLptMaxUsers) {
    for (int64_t u = tid; u < n_user; u += nt) {
      const int32_t Lu = s_len[u];
      int64_t rank = 0;
      for (int64_t w = 0; w < n_user; ++w) {
        const int32_t Lw = s_len[w];
        rank += (Lw > Lu) || (Lw == Lu && w < u);
      }
      order[rank] = (int32_t)u;
    }
  } else {
    for (int64_t u = tid; u < n_user; u += nt) order[u] = (int32_t)u;
  }
  __syncthreads();

  // 6. item counts per rank, prefix, emission --------------------------------
  // p.scratch holds 3 * n_user + 2 entries: order[n_user], then
  // items_before[n_user + 1], then units_before[n_user + 1].
  int32_t* items_before = p.scratch + n_user;
  int32_t* units_before = p.scratch + 2 * n_user + 1;   // n_user + 1 entries
  {
    int64_t carry_i = 0, carry_u = 0;
    for (int64_t base = 0; base < n_user; base += nt) {
      const int64_t rk = base + tid;
      int64_t ni = 0, nu = 0;
      if (rk < n_user) {
        const int32_t u = order[rk];
        const int64_t r = cand_start[u + 1] - cand_start[u];
        const int64_t L = off[u + 1] - off[u];
        if (r > 0 && L > 0) {
          const int64_t nmt = ceil_div64(r, cpt);
          const int64_t kt = ceil_div64(L, bn);
          const int64_t s = split_tiles ? ceil_div64(kt, split_tiles) : 1;
          ni = p.H * nmt * s;
          nu = s > 1 ? p.H * nmt : 0;
        }
      }
      int64_t tot_i, tot_u;
      const int64_t ex_i = block_exclusive_scan(ni, s_scan, &tot_i);
      const int64_t ex_u = block_exclusive_scan(nu, s_scan, &tot_u);
      if (rk < n_user) {
        items_before[rk] = (int32_t)(carry_i + ex_i);
        units_before[rk] = (int32_t)(carry_u + ex_u);
      }
      carry_i += tot_i;
      carry_u += tot_u;
    }
    if (tid == 0) {
      items_before[n_user] = (int32_t)carry_i;
      units_before[n_user] = (int32_t)carry_u;
    }
  }
  __syncthreads();
  const int64_t n_items = items_before[n_user];
  const int64_t n_units = units_before[n_user];
  if (n_items > p.max_items || n_units > p.max_units ||
      (split_tiles && n_items > p.max_split_items)) {
    // Cannot happen with the host's capacity bounds; refuse rather than overrun.
    if (tid == 0) {
      p.header->n_items = 0;
      p.header->error = kErrTimeout;
      atomicOr(p.err_word, kErrTimeout);
    }
    return;
  }
  // One warp per user rank: the user's sizes are read once, then its items
  // (consecutive in the list) are made 32 at a time, lane l the l-th, and
  // written by the warp as one contiguous run of 8-byte words.  (Item by
  // item, each thread searching and loading the user's sizes anew and
  // storing its 40 bytes word by word, this step took ~20 us for 4600 items:
  // one SM's store unit is the limit for scattered 4-byte stores.)
  static_assert(sizeof(WorkItem) == 40, "five 8-byte words per item");
  const int lane = tid & 31, nwarps = nt >> 5;
  for (int64_t rk = tid >> 5; rk < n_user; rk += nwarps) {
    const int64_t i0 = items_before[rk], i1 = items_before[rk + 1];
    if (i1 == i0) continue;
    const int32_t u = order[rk];
    const int64_t r = cand_start[u + 1] - cand_start[u];
    const int64_t L = off[u + 1] - off[u];
    const int64_t nmt = ceil_div64(r, cpt);
    const int64_t kt = ceil_div64(L, bn);
    const int64_t s = split_tiles ? ceil_div64(kt, split_tiles) : 1;
    for (int64_t ib = i0; ib < i1; ib += 32) {
      const int cnt = int(i1 - ib < 32 ? i1 - ib : 32);
      const int64_t i = ib + lane;
      WorkItem w = {};
      if (lane < cnt) {
        const int64_t local = i - i0;
        const int64_t split = local % s;
        const int64_t rest = local / s;
        const int64_t mt = rest % nmt;
        const int64_t h = rest / nmt;
        w.q_row = -1;
        w.n_split = (int32_t)s;
        w.user = u;
        w.head = (int32_t)h;
        w.cand_begin = (int32_t)(cand_start[u] + mt * cpt);
        w.n_cand = (int32_t)min((int64_t)cpt, r - mt * cpt);
        const int64_t kchunk = s > 1 ? split_tiles * bn : L;
        w.kv_begin = (int32_t)(off[u] + split * kchunk);
        w.kv_len = (int32_t)min(kchunk, L - split * kchunk);
        if (s > 1) {
          w.unit = (int32_t)(units_before[rk] + rest);
          w.unit_first = (int32_t)(i - split);
          if (split == 0) {
            p.units[w.unit].n_split = (int32_t)s;
            p.units[w.unit].arrived = 0;
          }
        } else {
          w.unit = -1;
          w.unit_first = (int32_t)i;
        }
      }
      // word j of the run is word j % 5 of lane j / 5's item
      uint32_t wv[10];
      memcpy(wv, &w, sizeof w);
      uint2* dst = reinterpret_cast<uint2*>(p.items + ib);   // 8-byte aligned: 40 * ib bytes in
#pragma unroll
      for (int t = 0; t < 5; ++t) {
        const int j = lane + 32 * t;
        const int src = j / 5, q = j % 5;
        uint2 v = make_uint2(0u, 0u);
#pragma unroll
        for (int x = 0; x < 5; ++x) {
          const uint32_t lo = __shfl_sync(0xffffffffu, wv[2 * x], src);
          const uint32_t hi = __shfl_sync(0xffffffffu, wv[2 * x + 1], src);
          if (q == x) v = make_uint2(lo, hi);
        }
        if (j < 5 * cnt) dst[j] = v;
      }
    }
  }
  // 7. tensor maps and header ------------------------------------------------
  const int32_t T = off[n_user];
  if (x.patch_maps && tid < 2) {
    // Copy the host-encoded template (row count unknown on the host) and set
    // its row count to T with tensormap.replace, then release it to the
    // tensor-map proxy of the GPU.
    const CUtensorMap* src = tid == 0 ? &x.kmap_tmpl : &x.vmap_tmpl;
    CUtensorMap* dst = tid == 0 ? x.kmap_dst : x.vmap_dst;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(CUtensorMap) / 16); ++i) d4[i] = s4[i];
    const int32_t rows = T > 0 ? T : 1;
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;"
                 :: "l"(dst), "r"(rows) : "memory");
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  }
  if (tid == 0) {
    p.header->n_items = (int32_t)n_items;
    p.header->sorted = sorted ? 1 : 0;
    p.header->total_keys = T;
    p.header->split_tiles = (int32_t)split_tiles;
    p.header->work_counter = 0;
    p.header->n_units = (int32_t)n_units;
    p.header->error = 0;
  }
}

}  // namespace ikbo
