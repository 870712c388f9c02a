// conv2tap.cu -- two-tap dynamic depthwise convolution ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Local Convolution": Conv_k(x)_t = k_{t,0} (.) x_t +
// k_{t,1} (.) x_{t-1}; each coefficient is a learned base kernel plus a small
// correction computed from the current hidden state, shared by every 16
// channels; the first position reads the last verified token's representation).
//
//   [c0; c1][m, :] = W_c h[m, :] (+ b_c)            W_c: [2G, d], G = d / 16
//   y[m, ch] = (k0[ch] + c0[m, ch/16]) x[m, ch] + (k1[ch] + c1[m, ch/16]) xp[ch]
//
// One fused kernel: the correction is a [M, d] x [d, 2G] contraction on the
// tensor cores (tcgen05 GEMM, fp32 accumulator in TMEM).  A CTA owns 128
// positions x 32 groups: its B tile is W_c rows [g0, g0+32) (-> c0) stacked on
// rows [G+g0, G+g0+32) (-> c1), so both coefficients of its 512 channels meet in
// one accumulator.  The epilogue parks the 64 correction columns in shared
// memory and then sweeps the 128 x 512 channel tile with coalesced 16-byte
// loads of x_t / x_{t-1} and 16-byte stores of y; the correction never leaves
// the SM.
#include "common.cuh"
#include "gemm_tc.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

struct ConvEpi {
  struct Params {
    const uint16_t* x;        // [M, d]
    const uint16_t* x_prev;   // [B, d]
    const uint16_t* k0;       // [d]
    const uint16_t* k1;       // [d]
    const float* b_c;         // [2G] or null
    void* y;                  // [M, d] bf16 or fp32
    int y_is_fp32;
    int M, L, d, G;
  };
  static constexpr int kGroups = 32;            // groups per CTA (512 channels)
  static constexpr int kBN = 2 * kGroups;       // c0 | c1 columns
  static constexpr int kPitch = kBN + 1;        // fp32 words per row in shared memory
  static constexpr int kSmemBytes = 128 * kPitch * 4;

  __device__ static void load_b(void* dst, const CUtensorMap* tm, int k, const Params& p, uint64_t* bar,
                                uint64_t pol) {
    const int g0 = blockIdx.y * kGroups;
    tma_load_2d(dst, tm, k, g0, bar, pol);                                             // c0 rows
    tma_load_2d(static_cast<uint8_t*>(dst) + kGroups * kTileRowBytes, tm, k, p.G + g0, bar, pol);  // c1 rows
  }

  __device__ static void consume(const Params& p, uint8_t* smem, int, int row_local, int c, const float (&v)[32]) {
    float* csm = reinterpret_cast<float*>(smem) + row_local * kPitch + c * kGroups;
    const int g0 = blockIdx.y * kGroups;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int g = g0 + i;
      float bias = 0.0f;
      if (p.b_c && g < p.G) bias = p.b_c[c * p.G + g];
      csm[i] = v[i] + bias;
    }
  }

  // All 192 threads sweep the 128 x (16 * ng) channel tile in 8-channel vectors;
  // each thread issues the loads of kUnroll vectors before using any of them.
  static constexpr int kUnroll = 4;

  __device__ static void finish(const Params& p, uint8_t* smem, int m0, int tid) {
    const float* csm = reinterpret_cast<const float*>(smem);
    const int g0 = blockIdx.y * kGroups;
    const int ng = (p.G - g0 < kGroups) ? p.G - g0 : kGroups;
    const int vec_per_row = 2 * ng;                 // 8-channel vectors per row
    const int rows = (p.M - m0 < 128) ? p.M - m0 : 128;
    const int total = rows * vec_per_row;
    for (int e0 = tid; e0 < total; e0 += kUnroll * kGemmThreads) {
      uint4 xv[kUnroll], pv[kUnroll], a0v[kUnroll], a1v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int e = e0 + u * kGemmThreads;
        if (e >= total) continue;
        const int r = e / vec_per_row, cv = e % vec_per_row;
        const int m = m0 + r;
        const int64_t ch = static_cast<int64_t>(g0) * 16 + cv * 8;
        const int t = m % p.L;
        const uint16_t* prow = t > 0 ? p.x + static_cast<int64_t>(m - 1) * p.d : p.x_prev + (m / p.L) * static_cast<int64_t>(p.d);
        xv[u] = *reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(m) * p.d + ch);
        pv[u] = *reinterpret_cast<const uint4*>(prow + ch);
        a0v[u] = __ldg(reinterpret_cast<const uint4*>(p.k0 + ch));
        a1v[u] = __ldg(reinterpret_cast<const uint4*>(p.k1 + ch));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int e = e0 + u * kGemmThreads;
        if (e >= total) continue;
        const int r = e / vec_per_row, cv = e % vec_per_row;
        const int m = m0 + r;
        const int gl = cv >> 1;
        const int64_t ch = static_cast<int64_t>(g0) * 16 + cv * 8;
        const float c0 = csm[r * kPitch + gl];
        const float c1 = csm[r * kPitch + kGroups + gl];
        const uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
        const uint32_t pw[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
        const uint32_t k0w[4] = {a0v[u].x, a0v[u].y, a0v[u].z, a0v[u].w};
        const uint32_t k1w[4] = {a1v[u].x, a1v[u].y, a1v[u].z, a1v[u].w};
        float out[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int sh = h * 16;
            const float xt = bf16_bits_to_float((xw[q] >> sh) & 0xFFFFu);
            const float xp = bf16_bits_to_float((pw[q] >> sh) & 0xFFFFu);
            const float a0 = bf16_bits_to_float((k0w[q] >> sh) & 0xFFFFu) + c0;
            const float a1 = bf16_bits_to_float((k1w[q] >> sh) & 0xFFFFu) + c1;
            out[2 * q + h] = fmaf(a0, xt, a1 * xp);
          }
        }
        const int64_t o = static_cast<int64_t>(m) * p.d + ch;
        if (p.y_is_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.y) + o);
          dst[0] = make_float4(out[0], out[1], out[2], out[3]);
          dst[1] = make_float4(out[4], out[5], out[6], out[7]);
        } else {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(out[2 * q]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(out[2 * q + 1]));
            w[q] = lo | (hi << 16);
          }
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.y) + o) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
};

}  // namespace

cudaError_t launch_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* hs,
                            const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                            const float* b_c, int64_t B, int64_t L, int64_t d, void* y,
                            int y_is_fp32, uint32_t* err, cudaStream_t stream) {
  const int64_t M = B * L;
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int64_t G = d / 16;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, hs ? hs : x, M, d, d, 128) ||
      !make_tmap_bf16_2d(&tb, W_c, 2 * G, d, d, ConvEpi::kGroups))
    return cudaErrorInvalidValue;
  ConvEpi::Params p{x, x_prev, k0, k1, b_c, y, y_is_fp32, static_cast<int>(M), static_cast<int>(L),
                    static_cast<int>(d), static_cast<int>(G)};
  const int grid_n = static_cast<int>((G + ConvEpi::kGroups - 1) / ConvEpi::kGroups);
  return launch_tc_gemm<ConvEpi::kBN, 3, ConvEpi>(ta, tb, static_cast<int>(M), static_cast<int>(d), grid_n, p,
                                                  err, stream);
}

}  // namespace dflash2
