// Explicit-broadcast comparison path: materialise each candidate's copy of
// its user's K and V, the system-level broadcast that "In-Kernel Broadcast
// Optimization", §1.4 item 1 and §3.1 (Fig. 10, left) describe as the
// conventional route.  Kept only so the two routes can be timed side by side.
#pragma once

#include "ikbo_common.cuh"

namespace ikbo {

// dst rows [dst_off[i], dst_off[i+1]) <- src rows [src_row[i], src_row[i] + len_i)
// for i in [0, n), rows of `row_bytes` bytes (a multiple of 16), for K and V.
__global__ void __launch_bounds__(256)
ikbo_broadcast_copy_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                           uint4* __restrict__ kb, uint4* __restrict__ vb,
                           const int32_t* __restrict__ src_row, const int64_t* __restrict__ dst_off,
                           int32_t n, int32_t row_vecs) {
  for (int32_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int64_t d0 = dst_off[i];
    const int64_t len = dst_off[i + 1] - d0;
    const int64_t s0 = src_row[i];
    const int64_t total = len * row_vecs;
    const uint4* ks = k + s0 * row_vecs;
    const uint4* vs = v + s0 * row_vecs;
    uint4* kd = kb + d0 * row_vecs;
    uint4* vd = vb + d0 * row_vecs;
    for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
      kd[e] = ks[e];
      vd[e] = vs[e];
    }
  }
}

}  // namespace ikbo
