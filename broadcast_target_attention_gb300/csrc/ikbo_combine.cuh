// Split-KV merge of the partial results of one (user, head, query tile).
//
// Each split item leaves, per query row, its unnormalised output O_s, its
// running maximum m_s (base 2) and its row sum l_s.  The exact result is
//   M = max_s m_s,  l = sum_s 2^(m_s - M) l_s,  out = sum_s 2^(m_s - M) O_s / l,
// the log-sum-exp merge of "Chapter 4: High-performance Kernels", §4.6.4
// (Flash-Decoding: lse = log sum_c exp(lse_c), o = sum_c exp(lse_c - lse) o_c),
// written with the (m, l) pair instead of lse = m + log l.
//
// The CTA that completes the last split of a unit does the merge: every split
// publishes its partial, fences, and increments the unit's arrival counter;
// the one that sees n_split - 1 is last.  Nobody waits, so an odd or single
// split can never stall the others.  This is the release/acquire hand-off of
// "In-Kernel Broadcast Optimization", Appendix 7, without its polling loop.
#pragma once

#include "ikbo_common.cuh"

namespace ikbo {

// Called by all `nthreads` threads (a multiple of 32, starting at thread
// `tid0`) of the CTA after the item's partial has been written.  Returns
// true in the CTA that merged.  `bar_id` is a named barrier for these threads.
template <int D>
__device__ __forceinline__ void merge_unit(const AttnParams& p, const WorkItem& w, int rows,
                                           int tid, int nthreads) {
  const int n_split = p.units[w.unit].n_split;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = nthreads >> 5;
  constexpr int kPer = D / 32;   // columns per lane
  for (int r = warp; r < rows; r += nwarps) {
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) {
      const float2 ml = __ldcg(&p.partial_ml[(int64_t)(w.unit_first + s) * kTileM + r]);
      M = fmaxf(M, ml.x);
    }
    float l = 0.f;
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    for (int s = 0; s < n_split; ++s) {
      const int64_t slot = (int64_t)(w.unit_first + s) * kTileM + r;
      const float2 ml = __ldcg(&p.partial_ml[slot]);
      const float a = fast_exp2(ml.x - M);
      l += a * ml.y;
      const float* o = p.partial_o + slot * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 x2 = __ldcg(reinterpret_cast<const float2*>(o + e));
        acc[e] += a * x2.x;
        acc[e + 1] += a * x2.y;
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int i = r / p.Lq, t = r - i * p.Lq;
    const int32_t g = w.cand_begin + i;
    const int64_t c = p.header->sorted ? g : p.perm[g];
    uint16_t* dst = p.out + (((c * p.H + w.head) * (int64_t)p.Lq + t) * D) + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const uint32_t lo = f32_to_bf16_rn(acc[e] * inv), hi = f32_to_bf16_rn(acc[e + 1] * inv);
      *reinterpret_cast<uint32_t*>(dst + e) = lo | (hi << 16);
    }
  }
}

}  // namespace ikbo
