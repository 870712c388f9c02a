// conv2tap.cu -- two-tap dynamic depthwise convolution ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Local Convolution": Conv_k(x)_t = k_{t,0} (.) x_t +
// k_{t,1} (.) x_{t-1}; each coefficient is a learned base kernel plus a small
// correction computed from the current hidden state, shared by every 16
// channels; the first position reads the last verified token's representation).
//
//   [c0; c1][m, :] = W_c h[m, :] (+ b_c)            W_c: [2G, d], G = d / 16
//   y[m, ch] = (k0[ch] + c0[m, ch/16]) x[m, ch] + (k1[ch] + c1[m, ch/16]) xp[ch]
//
// Two kernels.
//   1. The correction, a [M, d] x [d, 2G] contraction, on CTA pairs
//      (gemm_pair.cuh): 256 positions x 2 BNG columns per pair tile in one
//      MMA per K step, whose B operand is W_c rows [g0, g0 + BNG) (c0, in CTA
//      rank 0) and [G + g0, G + g0 + BNG) (c1, in rank 1), K split ks ways;
//      each split stores its fp32 partial [M, 2G] to the workspace.  One MMA
//      per K step reads the A tile once (two sub-block MMAs read it twice).
//   2. The taps, a streaming pass (conv_tap_kernel): one thread per 8-channel
//      unit walks the L positions of one sequence, carrying x_t over as the
//      next position's x_{t-1} (x_prev at the first), and writes y with 16-byte
//      stores.  Its x, x_prev, k0 and k1 loads do not depend on the correction,
//      so they are issued before the wait on the GEMM (programmatic dependent
//      launch); after it the thread sums the ks partials of its group in split
//      order (the same result on every run) and applies the taps in fp32.
#include <mutex>

#include "common.cuh"
#include "gemm_pair.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

constexpr int kConvBNG = 128;       // groups per pair tile (one N = 256 MMA: c0 and c1 of 128 groups)
constexpr int kTapThreads = 128;    // 8-channel units per CTA
constexpr int kTapRows = 8;         // positions whose x a thread holds at once

struct ConvShape {
  static constexpr int kSubs = 1;
  struct Params {
    int G, BNG;
  };
  // rank 0 holds the c0 rows of the tile's groups, rank 1 their c1 rows (half = BNG)
  __device__ static int b_row(const Params& p, int n_tile, int, int rank, int) {
    return (rank ? p.G : 0) + n_tile * p.BNG;
  }
  // tile columns [c, c + 4): c0 of groups g0 + c.., or c1 of groups g0 + c - BNG..
  // (BNG and G are multiples of 4, so the four are all valid or all not)
  __device__ static bool valid(const Params& p, int n_tile, int c) {
    const int g = n_tile * p.BNG + (c < p.BNG ? c : c - p.BNG);
    return g < p.G;
  }
  __device__ static int out_col(const Params& p, int n_tile, int c) {
    return c < p.BNG ? n_tile * p.BNG + c : p.G + n_tile * p.BNG + (c - p.BNG);
  }
};

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Packed fp32 pairs (Blackwell's f32x2 arithmetic: two independent fp32
// operations per instruction, each rounded as the scalar one would be).
// Element 0 of a pair sits in the low 32 bits.
__device__ __forceinline__ uint64_t pair(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(hi)) << 32 | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// one word of two bf16 values as a float pair
__device__ __forceinline__ uint64_t unpack2(uint32_t w) {
  return static_cast<uint64_t>(w & 0xFFFF0000u) << 32 | static_cast<uint64_t>(w << 16);
}

struct TapParams {
  const uint16_t* x;        // [M, d]
  const uint16_t* x_prev;   // [B, d]
  const uint16_t* k0;       // [d]
  const uint16_t* k1;       // [d]
  const float* b_c;         // [2G] or null
  const float* part;        // [ks, M, 2G]
  void* y;                  // [M, d] bf16 or fp32
  int y_is_fp32;
  int B, L, d, G, ks, units;   // units = d / 8 per position
};

// Grid (ceil(units / kTapThreads), B): thread -> unit u of sequence b.  KS =
// the number of K splits, so that a block's partial loads are all in flight
// before the first is used.  Five CTAs per SM (96 registers a thread) keep the
// 640 CTAs of 128 sequences at d = 5120 in one wave on 152 SMs.
template <int KS>
__global__ void __launch_bounds__(kTapThreads, 5) conv_tap_kernel(const TapParams p) {
  const int u = blockIdx.x * kTapThreads + threadIdx.x;
  const int b = blockIdx.y;
  const bool active = u < p.units;
  const int64_t M = static_cast<int64_t>(p.B) * p.L;
  const int64_t row0 = static_cast<int64_t>(b) * p.L;
  const int64_t ch = static_cast<int64_t>(u) * 8;
  const int g = u >> 1;
  // inputs that do not depend on the correction: in flight before the wait
  uint4 k0v = make_uint4(0, 0, 0, 0), k1v = k0v, prev = k0v;
  uint4 xs[kTapRows];
  const int n0 = p.L < kTapRows ? p.L : kTapRows;
  if (active) {
    k0v = __ldg(reinterpret_cast<const uint4*>(p.k0 + ch));
    k1v = __ldg(reinterpret_cast<const uint4*>(p.k1 + ch));
    prev = ldg_nc(p.x_prev + static_cast<int64_t>(b) * p.d + ch);
#pragma unroll
    for (int i = 0; i < kTapRows; ++i)
      if (i < n0) xs[i] = ldg_nc(p.x + (row0 + i) * p.d + ch);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (!active) return;
  const float bias0 = p.b_c ? p.b_c[g] : 0.0f, bias1 = p.b_c ? p.b_c[p.G + g] : 0.0f;
  const uint64_t k0p[4] = {unpack2(k0v.x), unpack2(k0v.y), unpack2(k0v.z), unpack2(k0v.w)};
  const uint64_t k1p[4] = {unpack2(k1v.x), unpack2(k1v.y), unpack2(k1v.z), unpack2(k1v.w)};
  const int64_t pstride = M * 2 * p.G;   // one split's partials
  for (int t0 = 0; t0 < p.L; t0 += kTapRows) {
    const int n = p.L - t0 < kTapRows ? p.L - t0 : kTapRows;
    // the rows' corrections: every partial of the block loaded first, then the
    // KS partials summed in split order, then the bias
    float q0[kTapRows][KS], q1[kTapRows][KS];
#pragma unroll
    for (int i = 0; i < kTapRows; ++i) {
      const float* pr = p.part + (row0 + t0 + (i < n ? i : 0)) * 2 * p.G;
#pragma unroll
      for (int qs = 0; qs < KS; ++qs) {
        q0[i][qs] = __ldcg(pr + qs * pstride + g);
        q1[i][qs] = __ldcg(pr + qs * pstride + p.G + g);
      }
    }
    float c0[kTapRows], c1[kTapRows];
#pragma unroll
    for (int i = 0; i < kTapRows; ++i) {
      float a0 = q0[i][0], a1 = q1[i][0];
#pragma unroll
      for (int qs = 1; qs < KS; ++qs) {
        a0 += q0[i][qs];
        a1 += q1[i][qs];
      }
      c0[i] = a0 + bias0;
      c1[i] = a1 + bias1;
    }
#pragma unroll
    for (int i = 0; i < kTapRows; ++i) {
      if (i >= n) break;
      const int64_t m = row0 + t0 + i;
      const uint4 xv = xs[i];
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      const uint32_t pw[4] = {prev.x, prev.y, prev.z, prev.w};
      const uint64_t c0p = pair(c0[i], c0[i]), c1p = pair(c1[i], c1[i]);
      uint64_t out[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        out[k] = fma2(add2(k0p[k], c0p), unpack2(xw[k]), mul2(add2(k1p[k], c1p), unpack2(pw[k])));
      const int64_t o = m * p.d + ch;
      if (p.y_is_fp32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.y) + o);
        __stcs(dst, make_uint4(static_cast<uint32_t>(out[0]), static_cast<uint32_t>(out[0] >> 32),
                               static_cast<uint32_t>(out[1]), static_cast<uint32_t>(out[1] >> 32)));
        __stcs(dst + 1, make_uint4(static_cast<uint32_t>(out[2]), static_cast<uint32_t>(out[2] >> 32),
                                   static_cast<uint32_t>(out[3]), static_cast<uint32_t>(out[3] >> 32)));
      } else {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(static_cast<uint32_t>(out[k])),
                                                          __uint_as_float(static_cast<uint32_t>(out[k] >> 32)));
          w[k] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.y) + o), make_uint4(w[0], w[1], w[2], w[3]));
      }
      prev = xv;
    }
    // the next block of positions
    if (t0 + kTapRows < p.L) {
      const int nn = p.L - t0 - kTapRows < kTapRows ? p.L - t0 - kTapRows : kTapRows;
#pragma unroll
      for (int i = 0; i < kTapRows; ++i)
        if (i < nn) xs[i] = ldg_nc(p.x + (row0 + t0 + kTapRows + i) * p.d + ch);
    }
  }
}

struct ConvPlan {
  PairGemmShape sh;
  int BNG;
};

ConvPlan conv_plan(int64_t M, int64_t d, int slots) {
  ConvPlan cp;
  const int G = static_cast<int>(d / 16);
  // N = 2 BNG = 32, 64 or 256: the pair-MMA widths that the parity tests cover
  // (a 96-group tile, N = 192, gave wrong rows in the second CTA of the pair).
  // A single row pair (at most 256 positions) takes 32-group tiles: more pairs
  // share W_c, which then dominates the bytes.
  cp.BNG = G <= 16 ? 16 : ((G <= 32 || M <= 256) ? 32 : kConvBNG);
  PairGemmShape& sh = cp.sh;
  sh.M = static_cast<int>(M);
  sh.K = static_cast<int>(d);
  sh.N = 2 * G;
  sh.BN = 2 * cp.BNG;
  sh.n_tiles = (G + cp.BNG - 1) / cp.BNG;
  sh.m_pairs = static_cast<int>((M + 255) / 256);
  sh.ks = pg_choose_ks(sh.n_tiles * sh.m_pairs, sh.K / kBK, slots);
  sh.tmem_cols = 32;
  while (sh.tmem_cols < static_cast<uint32_t>(sh.BN)) sh.tmem_cols <<= 1;
  return cp;
}

}  // namespace

size_t conv_workspace_bytes(int64_t B, int64_t L, int64_t d, int num_sms) {
  const int64_t M = B * L;
  const ConvPlan cp = conv_plan(M, d, num_sms);
  return static_cast<size_t>(cp.sh.ks) * static_cast<size_t>(M) * static_cast<size_t>(2 * (d / 16)) * sizeof(float);
}

cudaError_t launch_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* hs,
                            const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                            const float* b_c, int64_t B, int64_t L, int64_t d, void* y,
                            int y_is_fp32, void* workspace, uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t M = B * L;
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  // the plan depends on the SM count only (the workspace query sees the same one)
  ConvPlan cp = conv_plan(M, d, num_sms);
  if (!pg_plan(cp.sh)) return cudaErrorInvalidValue;
  const int G = static_cast<int>(d / 16);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, hs ? hs : x, M, d, d, 128) ||
      !make_tmap_bf16_2d(&tb, W_c, 2 * G, d, d, static_cast<uint32_t>(cp.BNG)))
    return cudaErrorInvalidValue;
  float* part = static_cast<float*>(workspace);
  cudaError_t e = launch_pair_gemm<ConvShape>(ta, tb, cp.sh, ConvShape::Params{G, cp.BNG}, part, err, stream);
  if (e != cudaSuccess) return e;
  TapParams tp{x, x_prev, k0, k1, b_c, part, y, y_is_fp32, static_cast<int>(B), static_cast<int>(L),
               static_cast<int>(d), G, cp.sh.ks, static_cast<int>(d / 8)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((d / 8 + kTapThreads - 1) / kTapThreads), static_cast<unsigned>(B), 1);
  cfg.blockDim = dim3(kTapThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (cp.sh.ks) {
    case 1: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<1>, tp);
    case 2: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<2>, tp);
    case 3: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<3>, tp);
    case 4: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<4>, tp);
    case 5: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<5>, tp);
    case 6: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<6>, tp);
    case 7: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<7>, tp);
    default: return cudaLaunchKernelEx(&cfg, conv_tap_kernel<8>, tp);
  }
}

}  // namespace dflash2
