// select.cu -- context gate and pairwise path-selector scores ("DFlash 2: Keep
// Drafting Parallel", "A Lightweight Path Selector", score equation
// S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>).
//
// gate_kernel      H = sigmoid(W_H h + b_H): one [B*L, d] x [d, 256] contraction,
//                  fp32 accumulate, sigmoid fused in the epilogue.
// pair_kernel      one CTA per block position (b, t): gathers the 16 predecessor
//                  rows of A and the 16 candidate rows of B (512 B each) with
//                  16-byte loads, forms G = A_pred (.) H_t in fp32 shared memory,
//                  and computes the 16 x 16 x 256 products with a 4 x 4 register
//                  tile per thread over 16 interleaved slices of r, reduced by a
//                  15-shuffle reduce-scatter.
#include "common.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

// ---------------------------------------------------------------------------
// gate: C[m, n] = sum_k h[m, k] W[n, k]; H = sigmoid(C + b)
// ---------------------------------------------------------------------------
constexpr int kGTileM = 64, kGTileN = 64, kGTileK = 32;

__global__ void __launch_bounds__(256) gate_kernel(const uint16_t* __restrict__ hs,
                                                   const uint16_t* __restrict__ W,
                                                   const float* __restrict__ bias, int64_t M,
                                                   int64_t d, float* __restrict__ gate) {
  __shared__ float As[kGTileK][kGTileM + 4];
  __shared__ float Ws[kGTileK][kGTileN + 4];
  const int tid = threadIdx.x;
  const int tm = tid >> 4, tn = tid & 15;          // 16 x 16 threads, 4 x 4 outputs each
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kGTileM;
  const int n0 = blockIdx.y * kGTileN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < d; k0 += kGTileK) {
    // 64 rows x 32 k of each operand: 256 threads x 8 elements (one 16-byte load)
    {
      const int r = tid >> 2, kc = (tid & 3) * 8;
      const int64_t gm = m0 + r;
      uint4 va = make_uint4(0, 0, 0, 0);
      if (gm < M) va = *reinterpret_cast<const uint4*>(hs + gm * d + k0 + kc);
      const uint4 vw = *reinterpret_cast<const uint4*>(W + static_cast<int64_t>(n0 + r) * d + k0 + kc);
      const uint32_t a[4] = {va.x, va.y, va.z, va.w}, w[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        As[kc + 2 * q][r] = bf16_bits_to_float(a[q] & 0xFFFFu);
        As[kc + 2 * q + 1][r] = bf16_bits_to_float(a[q] >> 16);
        Ws[kc + 2 * q][r] = bf16_bits_to_float(w[q] & 0xFFFFu);
        Ws[kc + 2 * q + 1][r] = bf16_bits_to_float(w[q] >> 16);
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kGTileK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tm * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = Ws[kk][tn * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jx = 0; jx < 4; ++jx) acc[i][jx] = fmaf(a[i], w[jx], acc[i][jx]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + tm * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int jx = 0; jx < 4; ++jx) {
      const int n = n0 + tn * 4 + jx;
      const float z = acc[i][jx] + (bias ? bias[n] : 0.0f);
      gate[gm * kEmbed + n] = 1.0f / (1.0f + expf(-z));
    }
  }
}

// ---------------------------------------------------------------------------
// pair scores
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pair_kernel(const int32_t* __restrict__ cand_idx,
                                                   const float* __restrict__ cand_val,
                                                   const int32_t* __restrict__ last_verified,
                                                   const float* __restrict__ gate,
                                                   const uint16_t* __restrict__ A,
                                                   const uint16_t* __restrict__ Bt, int64_t L,
                                                   int64_t V, float* __restrict__ S,
                                                   uint32_t* __restrict__ err) {
  __shared__ __align__(16) float G[kTopK][kEmbed];    // A[pred_i] (.) H_t
  __shared__ __align__(16) float Bc[kTopK][kEmbed];   // B[cand_j]
  __shared__ int32_t pred[kTopK], cur[kTopK];
  const int tid = threadIdx.x;
  const int64_t pos = blockIdx.x;              // b * L + t
  const int64_t b = pos / L, t = pos % L;
  if (tid < kTopK) {
    const int32_t p = (t == 0) ? last_verified[b] : cand_idx[(pos - 1) * kTopK + tid];
    pred[tid] = clamp_token(p, V, err);
    cur[tid] = clamp_token(cand_idx[pos * kTopK + tid], V, err);
  }
  __syncthreads();
  // 32 rows x 32 16-byte chunks = 1024 loads over 256 threads
  const float* Ht = gate + pos * kEmbed;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int e = tid + it * 256;
    const int row = e >> 5, ch = e & 31;       // rows 0..15: A, 16..31: B
    const bool isA = row < kTopK;
    const int r16 = row & (kTopK - 1);
    const uint16_t* src = isA ? A + static_cast<int64_t>(pred[r16]) * kEmbed
                              : Bt + static_cast<int64_t>(cur[r16]) * kEmbed;
    const uint4 v = *reinterpret_cast<const uint4*>(src + ch * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = bf16_bits_to_float(w[q] & 0xFFFFu);
      f[2 * q + 1] = bf16_bits_to_float(w[q] >> 16);
    }
    if (isA) {
      const float4 h0 = *reinterpret_cast<const float4*>(Ht + ch * 8);
      const float4 h1 = *reinterpret_cast<const float4*>(Ht + ch * 8 + 4);
      f[0] *= h0.x; f[1] *= h0.y; f[2] *= h0.z; f[3] *= h0.w;
      f[4] *= h1.x; f[5] *= h1.y; f[6] *= h1.z; f[7] *= h1.w;
      *reinterpret_cast<float4*>(&G[r16][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&G[r16][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      *reinterpret_cast<float4*>(&Bc[r16][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&Bc[r16][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
  __syncthreads();
  // thread = (block of 4 x 4 outputs, slice rs of r).  Slice rs owns the float4
  // chunks rs, rs + 16, rs + 32, rs + 48 of every row (conflict-free LDS.128).
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
  // reduce-scatter over the 16 slices (lane bits 0..3): lane rs ends with output rs
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

}  // namespace

cudaError_t launch_gate(const uint16_t* hs, const uint16_t* W_H, const float* b_H, int64_t M,
                        int64_t d, float* gate, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (d % kGTileK != 0) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>((M + kGTileM - 1) / kGTileM), kEmbed / kGTileN);
  gate_kernel<<<grid, 256, 0, stream>>>(hs, W_H, b_H, M, d, gate);
  return cudaGetLastError();
}

cudaError_t launch_pair_scores(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* last_verified, const float* gate, const uint16_t* A,
                               const uint16_t* Bt, int64_t B, int64_t L, int64_t V, float* S,
                               uint32_t* err, cudaStream_t stream) {
  pair_kernel<<<static_cast<unsigned>(B * L), 256, 0, stream>>>(cand_idx, cand_val, last_verified, gate,
                                                                A, Bt, L, V, S, err);
  return cudaGetLastError();
}

}  // namespace dflash2
