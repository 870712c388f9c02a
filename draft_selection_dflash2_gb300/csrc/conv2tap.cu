// conv2tap.cu -- two-tap dynamic depthwise convolution ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Local Convolution": Conv_k(x)_t = k_{t,0} (.) x_t +
// k_{t,1} (.) x_{t-1}; each coefficient is a learned base kernel plus a small
// correction computed from the current hidden state, shared by every 16
// channels; the first position reads the last verified token's representation).
//
//   [c0; c1][m, :] = W_c h[m, :] (+ b_c)            W_c: [2G, d], G = d / 16
//   y[m, ch] = (k0[ch] + c0[m, ch/16]) x[m, ch] + (k1[ch] + c1[m, ch/16]) xp[ch]
//
// One CTA owns one sequence b and a band of kGroups groups: it computes the
// 2 * kGroups correction columns it needs for all L positions (the correction
// never leaves shared memory), then applies the two-tap epilogue to the
// band's 16 * kGroups channels.
#include "common.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

constexpr int kGroups = 16;            // groups per CTA band -> 256 channels
constexpr int kCols = 2 * kGroups;     // correction columns per CTA
constexpr int kKTile = 64;
constexpr int kMaxConvL = 64;

__global__ void __launch_bounds__(256)
    conv2tap_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ x_prev,
                    const uint16_t* __restrict__ hs, const uint16_t* __restrict__ k0,
                    const uint16_t* __restrict__ k1, const uint16_t* __restrict__ W_c,
                    const float* __restrict__ b_c, int64_t L, int64_t d, void* __restrict__ y,
                    int y_is_fp32) {
  __shared__ float hsm[kMaxConvL][kKTile + 1];
  __shared__ float wsm[kCols][kKTile + 1];
  __shared__ float csm[kMaxConvL][kCols];
  const int tid = threadIdx.x;
  const int64_t b = blockIdx.y;
  const int64_t G = d / 16;
  const int64_t g0 = static_cast<int64_t>(blockIdx.x) * kGroups;
  const int ng = static_cast<int>(G - g0 < kGroups ? G - g0 : kGroups);
  const uint16_t* h = (hs ? hs : x) + b * L * d;

  // outputs (row, col) handled by this thread: col = tid % 32, rows tid/32 + 8 i
  const int col = tid & (kCols - 1);
  const int r0 = tid >> 5;
  float acc[kMaxConvL / 8];
#pragma unroll
  for (int i = 0; i < kMaxConvL / 8; ++i) acc[i] = 0.0f;
  // correction column -> W_c row: col < kGroups -> c0 group g0+col, else c1 group g0+col-kGroups
  const int cg = col < kGroups ? col : col - kGroups;
  const bool col_ok = cg < ng;
  const int64_t wrow = (col < kGroups ? 0 : G) + g0 + (col_ok ? cg : 0);

  for (int64_t kt = 0; kt < d; kt += kKTile) {
    for (int e = tid; e < L * kKTile; e += 256) {
      const int r = e / kKTile, k = e % kKTile;
      hsm[r][k] = bf16_bits_to_float(h[r * d + kt + k]);
    }
    for (int e = tid; e < kCols * kKTile; e += 256) {
      const int cc = e / kKTile, k = e % kKTile;
      const int cgg = cc < kGroups ? cc : cc - kGroups;
      const int64_t wr = (cc < kGroups ? 0 : G) + g0 + (cgg < ng ? cgg : 0);
      wsm[cc][k] = bf16_bits_to_float(W_c[wr * d + kt + k]);
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < kKTile; ++k) {
      const float w = wsm[col][k];
#pragma unroll
      for (int i = 0; i < kMaxConvL / 8; ++i) {
        const int r = r0 + 8 * i;
        if (r < L) acc[i] = fmaf(hsm[r][k], w, acc[i]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kMaxConvL / 8; ++i) {
    const int r = r0 + 8 * i;
    if (r < L) csm[r][col] = acc[i] + ((b_c && col_ok) ? b_c[wrow] : 0.0f);
  }
  __syncthreads();

  // epilogue: 16 * ng channels x L positions
  const int nch = 16 * ng;
  const int64_t ch0 = 16 * g0;
  for (int e = tid; e < L * nch; e += 256) {
    const int r = e / nch, cl = e % nch;
    const int64_t ch = ch0 + cl;
    const int g = cl >> 4;
    const int64_t m = b * L + r;
    const float xt = bf16_bits_to_float(x[m * d + ch]);
    const float xp = bf16_bits_to_float(r > 0 ? x[(m - 1) * d + ch] : x_prev[b * d + ch]);
    const float a0 = bf16_bits_to_float(k0[ch]) + csm[r][g];
    const float a1 = bf16_bits_to_float(k1[ch]) + csm[r][kGroups + g];
    const float v = fmaf(a0, xt, a1 * xp);
    if (y_is_fp32)
      static_cast<float*>(y)[m * d + ch] = v;
    else
      static_cast<__nv_bfloat16*>(y)[m * d + ch] = __float2bfloat16_rn(v);
  }
}

}  // namespace

cudaError_t launch_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* hs,
                            const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                            const float* b_c, int64_t B, int64_t L, int64_t d, void* y,
                            int y_is_fp32, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  if (L > kMaxConvL || d % kKTile != 0 || B > 65535) return cudaErrorInvalidValue;
  const int64_t G = d / 16;
  dim3 grid(static_cast<unsigned>((G + kGroups - 1) / kGroups), static_cast<unsigned>(B));
  conv2tap_kernel<<<grid, 256, 0, stream>>>(x, x_prev, hs, k0, k1, W_c, b_c, L, d, y, y_is_fp32);
  return cudaGetLastError();
}

}  // namespace dflash2
