// SIMT IKBO attention kernel: CUDA cores only, one warp per query row.
//
// An independent GPU implementation of the same work list as the tcgen05
// kernel, kept as a cross-check (selected with ikbo_set_kernel(1)).  Per
// query row it walks the item's key range with the online softmax of
// "Chapter 4: High-performance Kernels", §4.6.1 (running max, rescaled sum
// and output), in fp32, with scores in base 2.  The user's K/V rows are
// addressed through the work item -- no broadcast copy.
#pragma once

#include "ikbo_combine.cuh"
#include "ikbo_common.cuh"

namespace ikbo {

constexpr int kSimtThreads = 256;

template <int D>
__global__ void __launch_bounds__(kSimtThreads)
ikbo_attn_simt_kernel(const __grid_constant__ AttnParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kPer = D / 32;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  constexpr int nwarps = kSimtThreads / 32;
  __shared__ int s_last;
  const int n_items = p.header->n_items;
  const bool sorted = p.header->sorted != 0;

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkItem w = p.items[it];
    const int rows = w.n_cand * p.Lq;
    for (int r = warp; r < rows; r += nwarps) {
      const int i = r / p.Lq, t = r - i * p.Lq;
      const int32_t g = w.cand_begin + i;
      const int64_t c = sorted ? g : p.perm[g];
      const uint16_t* qrow = p.q + (((c * p.H + w.head) * (int64_t)p.Lq + t) * D) + lane * kPer;
      float qv[kPer];
#pragma unroll
      for (int e = 0; e < kPer; ++e) qv[e] = bf16_to_f32(qrow[e]) * p.scale_log2;
      float m = -INFINITY, l = 0.f;
      float acc[kPer];
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
      const int64_t rowstride = (int64_t)p.H * D;
      const uint16_t* kbase = p.k + (int64_t)w.kv_begin * rowstride + (int64_t)w.head * D + lane * kPer;
      const uint16_t* vbase = p.v + (int64_t)w.kv_begin * rowstride + (int64_t)w.head * D + lane * kPer;
      for (int j = 0; j < w.kv_len; ++j) {
        const uint16_t* kr = kbase + j * rowstride;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < kPer; ++e) s += qv[e] * bf16_to_f32(kr[e]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float m_new = fmaxf(m, s);
        const float alpha = fast_exp2(m - m_new);
        const float pj = fast_exp2(s - m_new);
        l = l * alpha + pj;
        const uint16_t* vr = vbase + j * rowstride;
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = acc[e] * alpha + pj * bf16_to_f32(vr[e]);
        m = m_new;
      }
      if (w.unit < 0) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t* dst = p.out + (((c * p.H + w.head) * (int64_t)p.Lq + t) * D) + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e) dst[e] = f32_to_bf16_rn(acc[e] * inv);
      } else {
        const int64_t slot = (int64_t)it * kTileM + r;
        float* o = p.partial_o + slot * D + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e) o[e] = acc[e];
        if (lane == 0) p.partial_ml[slot] = make_float2(m, l);
      }
    }
    if (w.unit >= 0) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(&p.units[w.unit].arrived, 1);
        s_last = prev == p.units[w.unit].n_split - 1;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        merge_unit<D>(p, w, rows, tid, kSimtThreads);
      }
    }
    __syncthreads();
  }
}

}  // namespace ikbo
