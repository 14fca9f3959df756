// IKBO target attention on the 5th-generation tensor cores (sm_103a):
// persistent, warp-specialised, TMA-fed, accumulators in tensor memory.
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
// the user's sequence is found through the work item (user_offsets), never
// through a per-candidate copy.  A tile that is only partly filled (odd or
// short groups, §3.2 "generalised" kernel) simply carries unused rows: the
// MMA computes them, the epilogue does not store them, and no warp waits for
// a partner that does not exist.
//
// Warp roles (one CTA per SM, 256 threads), after the Blackwell design of
// "Optimizing Jagged Flash Attention with TLX", §2.1 (dedicated load, MMA and
// softmax warps; explicit SMEM/TMEM buffers; S/P sharing one TMEM buffer, the
// PV accumulator its own; persistent CTAs):
//   warp 0      TMA producer: Q tile (double-buffered), then K_0, K_1, V_0,
//               K_2, V_1, ... into a ring of shared-memory slots;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               S_j = Q K_j^T (SS form, both operands in SMEM) into one of
//               two S buffers, then O += P_{j-1} V_{j-1} (TS form, P read
//               from TMEM), so S_j overlaps the softmax of tile j-1;
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

template <int D>
struct TcConfig {
  static constexpr int kCB = D / 64;                   // 128-byte column blocks per row
  static constexpr int kQBytes = kCB * kTileM * 128;    // one Q tile
  static constexpr int kKVBytes = kCB * kBlockN * 128;  // one K or V tile
  static constexpr int kNQ = 2;                         // Q buffers
  static constexpr int kNS = D == 128 ? 5 : 12;         // K/V ring slots
  static constexpr int kData = kNQ * kQBytes + kNS * kKVBytes;
  static constexpr int kNumBars = 2 * kNQ + 2 * kNS + 2 + 2 + 1 + 1;   // + tmem slot and flags
  static constexpr int kSmemBytes = kData + kNumBars * 8 + 64 + 1024;   // + flags, alignment
  // tensor-memory columns: two S/P buffers and the O accumulator
  static constexpr int kSCol = 0;
  static constexpr int kOCol = 2 * kBlockN;
  static constexpr int kTmemCols = 512;
  static_assert(kOCol + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Bounded mbarrier wait shared by all roles of a CTA.
struct Waiter {
  volatile int* abort;
  int* err_word;
  uint64_t timeout_ns;

  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    uint64_t t_end = 0;
    for (uint32_t spin = 1;; ++spin) {
      if (*abort) return false;
      if (ptx::mbar_try_wait(bar, parity)) return true;
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
  __device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) const {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait(bar, parity) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok != 0;
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Barrier of the four softmax warps built on a shared counter, bounded like
// every other wait (a hardware named barrier cannot time out, and a warp that
// aborted would leave the others stuck on it).  `target` grows by 4 per use.
__device__ __forceinline__ bool wg_sync(int* count, int target, const Waiter& W) {
  int ok = 1;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    atomicAdd(count, 1);
    uint64_t t_end = 0;
    for (uint32_t spin = 0; *reinterpret_cast<volatile int*>(count) < target; ++spin) {
      if (*W.abort) {
        ok = 0;
        break;
      }
      if ((spin & 63u) == 63u) {
        const uint64_t now = ptx::globaltimer();
        if (t_end == 0) {
          t_end = now + W.timeout_ns;
        } else if (now > t_end) {
          *W.abort = 1;
          atomicOr(W.err_word, kErrTimeout);
          ok = 0;
          break;
        }
      }
    }
    __threadfence_block();
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Split-KV merge of one query row by the CTA that finished the unit last
// (thread per row): M = max_s m_s, l = sum_s 2^(m_s - M) l_s,
// out = sum_s 2^(m_s - M) O_s / l  ("Chapter 4: High-performance Kernels",
// §4.6.4, log-sum-exp merge of Flash-Decoding).
template <int D>
__device__ __forceinline__ void merge_row(const AttnParams& p, const WorkItem& w, int row, int ci,
                                          int t, bool sorted) {
  const int ns = p.units[w.unit].n_split;
  const int64_t slot0 = (int64_t)w.unit_first * kTileM + row;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(&p.partial_ml[slot0 + (int64_t)s * kTileM]).x);
  float L = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float2 ml = __ldcg(&p.partial_ml[slot0 + (int64_t)s * kTileM]);
    L += fast_exp2(ml.x - M) * ml.y;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int32_t gpos = w.cand_begin + ci;
  const int64_t c = sorted ? gpos : p.perm[gpos];
  uint16_t* dst = p.out + (((c * p.H + w.head) * (int64_t)p.Lq + t) * D);
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 1
    for (int s0 = 0; s0 < ns; s0 += 2) {
      float a[2];
      float4 x[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int s = s0 + u;
        if (s < ns) {
          const int64_t slot = slot0 + (int64_t)s * kTileM;
          a[u] = fast_exp2(__ldcg(&p.partial_ml[slot]).x - M);
          const float4* src = reinterpret_cast<const float4*>(p.partial_o + slot * D + cc * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) x[u][q] = __ldcg(src + q);
        } else {
          a[u] = 0.f;
#pragma unroll
          for (int q = 0; q < 8; ++q) x[u][q] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[q * 4 + 0] += a[u] * x[u][q].x;
          acc[q * 4 + 1] += a[u] * x[u][q].y;
          acc[q * 4 + 2] += a[u] * x[u][q].z;
          acc[q * 4 + 3] += a[u] * x[u][q].w;
        }
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint4 v;
      v.x = pack_bf16(acc[q4 * 8 + 0] * inv, acc[q4 * 8 + 1] * inv);
      v.y = pack_bf16(acc[q4 * 8 + 2] * inv, acc[q4 * 8 + 3] * inv);
      v.z = pack_bf16(acc[q4 * 8 + 4] * inv, acc[q4 * 8 + 5] * inv);
      v.w = pack_bf16(acc[q4 * 8 + 6] * inv, acc[q4 * 8 + 7] * inv);
      d4[q4] = v;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
ikbo_attn_tc_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap qmap1) {
  using C = TcConfig<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  uint8_t* kv_smem = smem + C::kNQ * C::kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + C::kNQ;
  uint64_t* kv_full = q_empty + C::kNQ;
  uint64_t* kv_empty = kv_full + C::kNS;
  uint64_t* s_full = kv_empty + C::kNS;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* drain_bar = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_last = abort_flag + 1;
  int* wg_count = const_cast<int*>(s_last + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNQ; ++i) {
      ptx::mbar_init(ptx::smem_addr(&q_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&q_empty[i]), 1);
    }
    for (int i = 0; i < C::kNS; ++i) {
      ptx::mbar_init(ptx::smem_addr(&kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&s_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&p_full[i]), 4);
    }
    ptx::mbar_init(ptx::smem_addr(pv_done), 1);
    ptx::mbar_init(ptx::smem_addr(drain_bar), 1);
    *abort_flag = 0;
    *s_last = 0;
    *wg_count = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // Programmatic dependent launch: the planner may still be running; its
  // results (work list, patched tensor maps) are visible after this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t tmem = *tmem_slot;
  const int n_items = p.header->n_items;
  const bool sorted = p.header->sorted != 0;
  const Waiter W{abort_flag, p.err_word, p.timeout_ns};
  const int Lq = p.Lq;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::tensormap_acquire(p.kmap);
      ptx::tensormap_acquire(p.vmap);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      auto load_tile = [&](const void* map, int head, int32_t row) -> bool {
        const uint32_t slot = kv_it % C::kNS;
        if (!W.wait(ptx::smem_addr(&kv_empty[slot]), ((kv_it / C::kNS) & 1u) ^ 1u)) return false;
        const uint32_t bar = ptx::smem_addr(&kv_full[slot]);
        const uint32_t dst = ptx::smem_addr(kv_smem + slot * C::kKVBytes);
        ptx::mbar_arrive_expect_tx(bar, C::kKVBytes);
#pragma unroll
        for (int cb = 0; cb < C::kCB; ++cb)
          ptx::tma_load_2d(dst + cb * kBlockN * 128, map, bar, head * D + cb * 64, row);
        ++kv_it;
        return true;
      };
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = p.items[it];
        const int n = (w.kv_len + kBlockN - 1) / kBlockN;
        const uint32_t qb = q_it & 1u;
        if (!W.wait(ptx::smem_addr(&q_empty[qb]), ((q_it >> 1) & 1u) ^ 1u)) break;
        const uint32_t qbar = ptx::smem_addr(&q_full[qb]);
        const uint32_t qdst = ptx::smem_addr(q_smem + qb * C::kQBytes);
        if (!(p.debug_flags & 1)) {
          if (sorted) {
            const int nb = p.qbox;
            const int nbox = (w.n_cand + nb - 1) / nb;
            ptx::mbar_arrive_expect_tx(qbar, uint32_t(nbox * nb * Lq * 128 * C::kCB));
            for (int cb = 0; cb < C::kCB; ++cb)
              for (int b = 0; b < nbox; ++b)
                ptx::tma_load_4d(qdst + cb * kTileM * 128 + b * nb * Lq * 128, &qmap, qbar,
                                 cb * 64, 0, w.head, w.cand_begin + b * nb);
          } else {
            ptx::mbar_arrive_expect_tx(qbar, uint32_t(w.n_cand * Lq * 128 * C::kCB));
            for (int i = 0; i < w.n_cand; ++i) {
              const int32_t c = p.perm[w.cand_begin + i];
              for (int cb = 0; cb < C::kCB; ++cb)
                ptx::tma_load_4d(qdst + cb * kTileM * 128 + i * Lq * 128, &qmap1, qbar, cb * 64, 0,
                                 w.head, c);
            }
          }
        }
        ++q_it;
        // K/V tiles in the order the MMA warp consumes them: K0, K1, V0, K2, V1, ...
        for (int j = 0; j <= n && ok; ++j) {
          if (j < n) ok = load_tile(p.kmap, w.head, w.kv_begin + j * kBlockN);
          if (ok && j >= 1) ok = load_tile(p.vmap, w.head, w.kv_begin + (j - 1) * kBlockN);
        }
      }
      // Drain: every armed barrier phase must complete before the CTA exits.
      for (uint32_t s = 0; s < C::kNS && s < kv_it; ++s) {
        const uint32_t uses = (kv_it - s + C::kNS - 1) / C::kNS;
        W.drain(ptx::smem_addr(&kv_full[s]), (uses - 1) & 1u);
      }
      if (!(p.debug_flags & 1))
        for (uint32_t b = 0; b < C::kNQ && b < q_it; ++b) {
          const uint32_t uses = (q_it - b + 1) / 2;
          W.drain(ptx::smem_addr(&q_full[b]), (uses - 1) & 1u);
        }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kTileM, kBlockN, 0);
      constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kTileM, 64, 1);
      uint32_t kv_it = 0, q_it = 0, g = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = p.items[it];
        const int n = (w.kv_len + kBlockN - 1) / kBlockN;
        const uint32_t qb = q_it & 1u;
        if (!W.wait(ptx::smem_addr(&q_full[qb]), (q_it >> 1) & 1u)) break;
        ptx::tc_fence_after();
        const uint32_t q_base = ptx::smem_addr(q_smem + qb * C::kQBytes);
        for (int j = 0; j <= n; ++j) {
          if (j < n) {
            const uint32_t slot = kv_it % C::kNS;
            if (!W.wait(ptx::smem_addr(&kv_full[slot]), (kv_it / C::kNS) & 1u)) {
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
              const uint64_t b = ptx::smem_desc_sw128(k_base + cb * kBlockN * 128 + koff, 16, 1024);
              ptx::mma_ss(d_tmem, a, b, kIdescQK, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(ptx::smem_addr(&kv_empty[slot]));
            ptx::mma_commit(ptx::smem_addr(&s_full[sb]));
            if (j == n - 1) ptx::mma_commit(ptx::smem_addr(&q_empty[qb]));
            ++kv_it;
          }
          if (j >= 1) {
            const uint32_t pj = g + j - 1;
            const uint32_t pb = pj & 1u;
            if (!W.wait(ptx::smem_addr(&p_full[pb]), (pj >> 1) & 1u)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t slot = kv_it % C::kNS;
            if (!W.wait(ptx::smem_addr(&kv_full[slot]), (kv_it / C::kNS) & 1u)) {
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
                const uint64_t b = ptx::smem_desc_sw128(v_base + cb * kBlockN * 128 + kk * 16 * 128,
                                                        kBlockN * 128, 1024);
                ptx::mma_ts(tmem + C::kOCol + cb * 64, a_tmem + kk * 8, b, kIdescPV,
                            (j > 1 || kk > 0) ? 1u : 0u);
              }
            }
            ptx::mma_commit(ptx::smem_addr(&kv_empty[slot]));
            ptx::mma_commit(ptx::smem_addr(pv_done));
            ++kv_it;
          }
        }
        g += n;
        ++q_it;
      }
      // All issued MMAs must finish before tensor memory is released.
      ptx::mma_commit(ptx::smem_addr(drain_bar));
      W.drain(ptx::smem_addr(drain_bar), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------- softmax / correction / epilogue
    const int row = threadIdx.x - 128;                       // TMEM lane == tile row
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t g = 0, pv_it = 0;
    int wg_target = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const WorkItem w = p.items[it];
      const int n = (w.kv_len + kBlockN - 1) / kBlockN;
      const int rows = w.n_cand * Lq;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const uint32_t gj = g + j;
        const uint32_t sb = gj & 1u;
        if (!W.warp_wait(ptx::smem_addr(&s_full[sb]), (gj >> 1) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t scol = tmem + lane_off + C::kSCol + sb * kBlockN;
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(scol + c * 32, sr[c]);
        ptx::tmem_ld_wait();
        const int valid = min(kBlockN, w.kv_len - j * kBlockN);
        // row maximum of the scaled scores (of the raw minimum when scale < 0)
        const float sgn = sl2 < 0.f ? -1.f : 1.f;
        float mx = -INFINITY;
        if (valid == kBlockN) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, sgn * __uint_as_float(sr[c][e]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < valid) mx = fmaxf(mx, sgn * __uint_as_float(sr[c][e]));
        }
        mx *= sgn * sl2;
        const float m_new = (m == -INFINITY || mx > m + kLazyRescale) ? fmaxf(m, mx) : m;
        const float alpha = fast_exp2(m - m_new);   // 0 on the first tile, 1 when m stays
        float sum = 0.f;
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
            sum += p0 + p1;
            pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16(p0, p1);
          }
        l = l * alpha + sum;
        // P (bf16 pairs) overwrites the first half of this S buffer.
        ptx::tmem_st32(scol, pk[0]);
        ptx::tmem_st32(scol + 32, pk[1]);
        ptx::tmem_st_wait();
        if (j > 0) {
          // O holds P_0..P_{j-1} V: wait for PV_{j-1}, then rescale if m moved.
          if (!W.warp_wait(ptx::smem_addr(pv_done), pv_it & 1u)) {
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
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&p_full[sb]));
      }
      if (!ok) break;
      // ---- epilogue: O / l
      if (!W.warp_wait(ptx::smem_addr(pv_done), pv_it & 1u)) break;
      ++pv_it;
      ptx::tc_fence_after();
      const uint32_t ocol = tmem + lane_off + C::kOCol;
      const bool live = row < rows;
      const int ci = live ? row / Lq : 0;
      const int t = live ? row - ci * Lq : 0;
      if (w.unit < 0) {
        const int32_t gpos = w.cand_begin + ci;
        const int64_t c = live ? (sorted ? gpos : p.perm[gpos]) : 0;
        uint16_t* dst = p.out + (((c * p.H + w.head) * (int64_t)Lq + t) * D);
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + cc * 32, o);
          ptx::tmem_ld_wait();
          if (live) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
              d4[q4] = v;
            }
          }
        }
      } else {
        const int64_t slot = (int64_t)it * kTileM + row;
        float* po = p.partial_o + slot * D;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(ocol + cc * 32, o);
          ptx::tmem_ld_wait();
          if (live) {
            float4* d4 = reinterpret_cast<float4*>(po + cc * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              __stcg(d4 + q4, make_float4(__uint_as_float(o[q4 * 4 + 0]), __uint_as_float(o[q4 * 4 + 1]),
                                          __uint_as_float(o[q4 * 4 + 2]), __uint_as_float(o[q4 * 4 + 3])));
          }
        }
        if (live) __stcg(&p.partial_ml[slot], make_float2(m, l));
        __threadfence();
        if (!wg_sync(wg_count, wg_target += 4, W)) break;
        if (row == 0) {
          const int prev = atomicAdd(&p.units[w.unit].arrived, 1);
          *s_last = prev == p.units[w.unit].n_split - 1 ? 1 : 0;
        }
        if (!wg_sync(wg_count, wg_target += 4, W)) break;
        const bool last = *s_last != 0;
        if (!wg_sync(wg_count, wg_target += 4, W)) break;   // s_last may be reused after this
        if (last) {
          __threadfence();
          if (live) merge_row<D>(p, w, row, ci, t, sorted);
        }
      }
      g += n;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace ikbo
