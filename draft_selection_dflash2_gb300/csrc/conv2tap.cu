// conv2tap.cu -- two-tap dynamic depthwise convolution ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Local Convolution": Conv_k(x)_t = k_{t,0} (.) x_t +
// k_{t,1} (.) x_{t-1}; each coefficient is a learned base kernel plus a small
// correction computed from the current hidden state, shared by every 16
// channels; the first position reads the last verified token's representation).
//
//   [c0; c1][m, :] = W_c h[m, :] (+ b_c)            W_c: [2G, d], G = d / 16
//   y[m, ch] = (k0[ch] + c0[m, ch/16]) x[m, ch] + (k1[ch] + c1[m, ch/16]) xp[ch]
//
// One fused kernel (gemm_splitk.cuh): the correction is a [M, d] x [d, 2G]
// contraction on the tensor cores, tiled as 128 positions x BNG groups; the
// tile's B operand stacks W_c rows [g0, g0+BNG) (-> c0) on rows [G+g0, G+g0+BNG)
// (-> c1), so both coefficients of the tile's 16*BNG channels meet in one
// accumulator.  The K loop is split over a cluster of ks CTAs whose fp32
// partials meet through distributed shared memory.  Cluster rank r then owns
// 128/ks rows: it sums their slots once, and stages the rows' x_t in shared
// memory with bulk copies (all of them in one pass when they fit, as they do
// for d = 5120), together with the previous-tap rows that are not the row
// above (the pass's first row, and every first position, whose previous tap
// is x_prev[b]).  Every (row, 8 channels) item is then independent: its two
// taps come from shared memory (or, for consecutive rows of one thread, the
// register that held the row above), and y leaves with 16-byte stores.  The
// correction never leaves the SMs.
#include "common.cuh"
#include "gemm_splitk.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

constexpr int kMaxGroupsPerTile = 160;   // BN = 2 * BNG <= 320 (two N = 160 MMAs)
constexpr int kPrevTableBytes = 512;     // previous-tap row offsets of one pass (<= 128 rows), end of the region

struct ConvEpi {
  struct Params {
    const uint16_t* x;        // [M, d]
    const uint16_t* x_prev;   // [B, d]
    const uint16_t* k0;       // [d]
    const uint16_t* k1;       // [d]
    const float* b_c;         // [2G] or null
    void* y;                  // [M, d] bf16 or fp32
    int y_is_fp32;
    int M, L, d, G, BNG;
    int PR;                   // x_t rows per pass; the staged previous-tap rows follow them
    int stage_off;            // byte offset of the pass buffer in the region
  };

  __host__ __device__ static int sub_n(int BN) { return BN > 256 ? BN / 2 : BN; }

  __device__ static void load_b(void* dst, const CUtensorMap* tm, int k, int n_tile, const Params& p, uint64_t* bar,
                                uint64_t pol) {
    const int g0 = n_tile * p.BNG;
    tma_load_2d(dst, tm, k, g0, bar, pol);                                                // c0 rows
    tma_load_2d(static_cast<uint8_t*>(dst) + p.BNG * kTileRowBytes, tm, k, p.G + g0, bar, pol);  // c1 rows
  }

  // Staged previous-tap rows of a pass of n rows starting at row mb: the
  // pass's row 0, then every row j >= 1 at a first position ((mb + j) % L == 0),
  // in row order; prev_index(j) is such a row's place among them.
  __device__ static int staged_prev_count(int mb, int n, int L) { return 1 + (mb + n - 1) / L - mb / L; }
  __device__ static int prev_index(int mb, int j, int L) { return j == 0 ? 0 : 1 + (mb + j - 1) / L - mb / L; }

  __device__ static __forceinline__ void issue_pass(const Params& p, uint8_t* buf, uint64_t* bar, int mb, int n,
                                                    int g0, uint32_t cpy, uint64_t pol) {
    const int rowb = p.BNG * 32;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n + staged_prev_count(mb, n, p.L)) * cpy);
    const uint16_t* xs = p.x + static_cast<int64_t>(mb) * p.d + g0 * 16;   // row mb + j at xs + j * d
    int t = mb % p.L, b = mb / p.L, k = 1;                                    // position, sequence, next prev slot
    for (int j = 0; j < n; ++j) {
      bulk_g2s(buf + j * rowb, xs + static_cast<int64_t>(j) * p.d, cpy, bar, pol);
      if (t == 0 || j == 0) {
        const uint16_t* src = t == 0 ? p.x_prev + static_cast<int64_t>(b) * p.d + g0 * 16
                                     : xs + static_cast<int64_t>(j - 1) * p.d;
        bulk_g2s(buf + (p.PR + (j == 0 ? 0 : k++)) * rowb, src, cpy, bar, pol);
      }
      if (++t == p.L) {
        t = 0;
        ++b;
      }
    }
  }

  // Packed fp32 pairs (Blackwell's f32x2 arithmetic: two independent fp32
  // operations per instruction, each rounded as the scalar one would be).
  // Element 0 of a pair sits in the low 32 bits.
  __device__ static __forceinline__ uint64_t pair(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(hi)) << 32 | __float_as_uint(lo);
  }
  __device__ static __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
  }
  __device__ static __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
  }
  __device__ static __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
  }
  // one word of two bf16 values as a float pair
  __device__ static __forceinline__ uint64_t unpack2(uint32_t w) {
    return static_cast<uint64_t>(w & 0xFFFF0000u) << 32 | static_cast<uint64_t>(w << 16);
  }

  // y[m, ch .. ch+8) from 8 channels of x_t, x_{t-1}, the k0, k1 pairs and the
  // group's coefficients: (k0 + c0) x_t + (k1 + c1) x_{t-1}, in fp32.
  __device__ static __forceinline__ void write8(const Params& p, int64_t m, int64_t ch, uint4 xv, uint4 pv,
                                                const uint64_t (&k0p)[4], const uint64_t (&k1p)[4], float c0,
                                                float c1) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
    const uint64_t c0p = pair(c0, c0), c1p = pair(c1, c1);
    uint64_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      out[q] = fma2(add2(k0p[q], c0p), unpack2(xw[q]), mul2(add2(k1p[q], c1p), unpack2(pw[q])));
    const int64_t o = m * p.d + ch;
    if (p.y_is_fp32) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.y) + o);
      dst[0] = make_uint4(static_cast<uint32_t>(out[0]), static_cast<uint32_t>(out[0] >> 32),
                          static_cast<uint32_t>(out[1]), static_cast<uint32_t>(out[1] >> 32));
      dst[1] = make_uint4(static_cast<uint32_t>(out[2]), static_cast<uint32_t>(out[2] >> 32),
                          static_cast<uint32_t>(out[3]), static_cast<uint32_t>(out[3] >> 32));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(static_cast<uint32_t>(out[q])),
                                                        __uint_as_float(static_cast<uint32_t>(out[q] >> 32)));
        w[q] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.y) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }

  __device__ static __forceinline__ void finish(const Params& p, const SplitKShape& sh, uint8_t* region,
                                                uint64_t* bars, int m0, int n_tile, int rank, int tid, uint32_t* err) {
    const int rows_per = 128 / sh.ks;
    const int pitch = sk_partial_pitch(sh.BN);
    float* sums = reinterpret_cast<float*>(region);
    const int g0 = n_tile * p.BNG;
    const int ng = (p.G - g0 < p.BNG) ? p.G - g0 : p.BNG;
    const int mb = m0 + rank * rows_per;                       // this rank's first row
    const int nrows = p.M - mb >= rows_per ? rows_per : (p.M - mb > 0 ? p.M - mb : 0);

    // 1. slot 0 <- the sum of the slots (each element is read and written by one thread)
    if (sh.ks > 1) {
      const SkPartials parts(sums, sh.ks, pitch);
      const int c4n = sh.BN / 4;
      const int total = nrows * c4n;
      for (int e0 = tid; e0 < total; e0 += 2 * kSkThreads) {
        float4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = e0 + u * kSkThreads;
          if (e < total) v[u] = parts.sum4(e / c4n, (e % c4n) * 4);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = e0 + u * kSkThreads;
          if (e < total) *reinterpret_cast<float4*>(sums + (e / c4n) * pitch + (e % c4n) * 4) = v[u];
        }
      }
    }
    __syncthreads();   // the other slots are free from here on

    // 2. passes of up to PR rows through one buffer.  Thread -> 8-channel unit
    //    u = tid % 2ng (its k0, k1 and bias stay in registers) and rows
    //    j = tid / 2ng + i * R, R = threads / 2ng; with R == 1 (d = 5120) a thread
    //    walks consecutive rows and carries x_t over as the next row's x_{t-1}.
    uint8_t* buf = region + p.stage_off;
    int* prev_off = reinterpret_cast<int*>(region + sh.region_bytes - kPrevTableBytes);   // per row of a pass
    const int rowb = p.BNG * 32;
    const uint32_t cpy = static_cast<uint32_t>(ng) * 32;
    const int nu = 2 * ng;
    const int R = kSkThreads / nu;
    const bool active = tid < R * nu;
    const int u = tid % nu, r0 = tid / nu;
    uint4 k0v = make_uint4(0, 0, 0, 0), k1v = k0v;
    float b0 = 0.0f, b1 = 0.0f;
    if (active) {
      k0v = __ldg(reinterpret_cast<const uint4*>(p.k0 + static_cast<int64_t>(g0) * 16) + u);
      k1v = __ldg(reinterpret_cast<const uint4*>(p.k1 + static_cast<int64_t>(g0) * 16) + u);
      if (p.b_c) {
        b0 = p.b_c[g0 + (u >> 1)];
        b1 = p.b_c[p.G + g0 + (u >> 1)];
      }
    }
    const uint64_t k0p[4] = {unpack2(k0v.x), unpack2(k0v.y), unpack2(k0v.z), unpack2(k0v.w)};
    const uint64_t k1p[4] = {unpack2(k1v.x), unpack2(k1v.y), unpack2(k1v.z), unpack2(k1v.w)};
    bool ok = true;
    for (int pass = 0, lr0 = 0; lr0 < nrows; ++pass, lr0 += p.PR) {
      const int n = nrows - lr0 < p.PR ? nrows - lr0 : p.PR;
      const int mp = mb + lr0;
      if (tid == 0 && ok) issue_pass(p, buf, &bars[0], mp, n, g0, cpy, l2_policy_evict_first());
      if (tid < n)   // staged previous-tap row of row tid, or -1 for the row above
        prev_off[tid] = (tid == 0 || (mp + tid) % p.L == 0) ? (p.PR + prev_index(mp, tid, p.L)) * rowb : -1;
      ok = ok && mbar_wait_bounded(&bars[0], pass & 1, err);
      __syncthreads();   // the pass's rows and the row table are in place
      if (ok && active) {
        uint4 carry = make_uint4(0, 0, 0, 0);
        for (int jb = r0; jb < n; jb += 4 * R) {
          uint4 xv[4], pv[4];
          float c0[4], c1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = jb + i * R;
            if (j >= n) break;
            xv[i] = reinterpret_cast<const uint4*>(buf + j * rowb)[u];
            const int po = prev_off[j];
            if (po >= 0)
              pv[i] = reinterpret_cast<const uint4*>(buf + po)[u];
            else if (R == 1)
              pv[i] = i == 0 ? carry : xv[i - 1];
            else
              pv[i] = reinterpret_cast<const uint4*>(buf + (j - 1) * rowb)[u];
            const float* srow = sums + (lr0 + j) * pitch;
            c0[i] = srow[u >> 1] + b0;
            c1[i] = srow[p.BNG + (u >> 1)] + b1;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = jb + i * R;
            if (j >= n) break;
            write8(p, mp + j, static_cast<int64_t>(g0) * 16 + u * 8, xv[i], pv[i], k0p, k1p, c0[i], c1[i]);
            carry = xv[i];
          }
        }
      }
      __syncthreads();   // the buffer and the table are free again
    }
  }
};

}  // namespace

cudaError_t launch_conv2tap(const uint16_t* x, const uint16_t* x_prev, const uint16_t* hs,
                            const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c,
                            const float* b_c, int64_t B, int64_t L, int64_t d, void* y,
                            int y_is_fp32, uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t M = B * L;
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int G = static_cast<int>(d / 16);
  int BNG = (G + 15) / 16 * 16;
  if (BNG > kMaxGroupsPerTile) BNG = kMaxGroupsPerTile;
  SplitKShape sh;
  sh.M = static_cast<int>(M);
  sh.K = static_cast<int>(d);
  sh.BN = 2 * BNG;
  sh.n_tiles = (G + BNG - 1) / BNG;
  sh.m_tiles = static_cast<int>((M + 127) / 128);
  sh.ks = sk_choose_ks(sh.n_tiles * sh.m_tiles, sh.K / kBK, num_sms);
  sh.tmem_cols = 32;
  while (sh.tmem_cols < static_cast<uint32_t>(sh.BN)) sh.tmem_cols <<= 1;
  if (!sk_plan(sh)) return cudaErrorInvalidValue;
  // the pass buffer follows the summed slot rows: PR x_t rows, then room for the
  // staged previous-tap rows of any PR consecutive rows
  const int stage_off = ((128 / sh.ks) * sk_partial_pitch(sh.BN) * 4 + 127) / 128 * 128;
  const int rowb = BNG * 32;
  const int Li = static_cast<int>(L < 128 ? L : 128);
  int PR = 128 / sh.ks;
  auto prevs = [&](int r) { const int c = 1 + (r - 1 + Li - 1) / Li; return c < r ? c : r; };
  while (PR > 0 && (PR + prevs(PR)) * rowb > sh.region_bytes - kPrevTableBytes - stage_off) --PR;
  if (PR < 1) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, hs ? hs : x, M, d, d, 128) || !make_tmap_bf16_2d(&tb, W_c, 2 * G, d, d, BNG))
    return cudaErrorInvalidValue;
  ConvEpi::Params p{x, x_prev, k0, k1, b_c, y, y_is_fp32, static_cast<int>(M), static_cast<int>(L),
                    static_cast<int>(d), G, BNG, PR, stage_off};
  return launch_splitk_gemm<ConvEpi>(ta, tb, sh, p, err, stream);
}

}  // namespace dflash2
