// pair_math.cuh -- the 16 x 16 pair products of one block position, shared by
// the table-form and the projection-form pair kernels ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector"):
//   S[pos, i, j] = U[pos, j] + sum_r G[i][r] * Bc[j][r]
// with G = A(pred) (.) H_t and Bc = B(cand) already in fp32 shared memory.
#pragma once

#include "common.cuh"

namespace dflash2 {

// 256 threads.  Thread = (block of 4 x 4 outputs, slice rs of r); slice rs owns
// the float4 chunks rs, rs + 16, rs + 32, rs + 48 of every row (conflict-free
// LDS.128), and a 15-shuffle reduce-scatter over the 16 slices leaves output rs
// in lane rs of each group.
__device__ __forceinline__ void pair_products(const float (*G)[kEmbed], const float (*Bc)[kEmbed],
                                              const float* __restrict__ cand_val, float* __restrict__ S,
                                              int64_t pos, int tid) {
  const int rs = tid & 15, blk = tid >> 4;
  const int ib = blk >> 2, jb = blk & 3;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int c = rs + 16 * m;
    float4 g[4], bb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) g[i] = *reinterpret_cast<const float4*>(&G[4 * ib + i][4 * c]);
#pragma unroll
    for (int jx = 0; jx < 4; ++jx) bb[jx] = *reinterpret_cast<const float4*>(&Bc[4 * jb + jx][4 * c]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jx = 0; jx < 4; ++jx) {
        float a = acc[i * 4 + jx];
        a = fmaf(g[i].x, bb[jx].x, a);
        a = fmaf(g[i].y, bb[jx].y, a);
        a = fmaf(g[i].z, bb[jx].z, a);
        a = fmaf(g[i].w, bb[jx].w, a);
        acc[i * 4 + jx] = a;
      }
  }
#pragma unroll
  for (int half = 8; half >= 1; half >>= 1) {
    const bool upper = (rs & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? acc[i] : acc[i + half];
      const float keep = upper ? acc[i + half] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, half);
    }
  }
  const int i = 4 * ib + (rs >> 2), j = 4 * jb + (rs & 3);
  S[(pos * kTopK + i) * kTopK + j] = cand_val[pos * kTopK + j] + acc[0];
}

}  // namespace dflash2
