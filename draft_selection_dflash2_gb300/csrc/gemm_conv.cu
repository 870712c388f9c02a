// gemm_conv.cu -- the two-tap dynamic conv of "A Lightweight Local Convolution"
// ("DFlash 2: Keep Drafting Parallel") fused into the GEMM that produces its
// input, the output projection of a drafter sublayer, so x never goes to memory:
//   x = A W^T                      (tensor cores, fp32, not rounded)
//   c = W_c h + b_c                (correction from a given hidden state)
//   y_t = (k0 + c0_t) x_t + (k1 + c1_t) x_{t-1},   x_{-1} = x_prev
//
// gemm_conv_kernel: one persistent cooperative launch, one CTA per SM, over two
// kinds of 128 x 320 tiles (320 = 2 x 160-column MMAs; 5120 = 16 x 320, so a
// [2048, 5120] output is 256 tiles, two rounds on 152 SMs).  Rows are tiled in
// whole blocks, R = floor(128 / L) * L per tile, so x_{t-1} of every row but a
// block's first lies in the same tile.
//   correction tiles (first in the tile order): c = h W_c^T + b_c for a row
//     tile and 320 of the 2d/16 correction columns, stored as fp32 in the
//     caller's workspace; the row tile's counter is then raised (release).
//   main tiles: x = A W^T for a row tile and 320 channels; the epilogue waits
//     (acquire, bounded) until the row tile's corrections are all stored.
//   warp 0      TMA producer: a 128 x 64 tile of A (or h) and two 160 x 64
//               tiles of W (or W_c) per stage, 4-deep ring of 56 KB stages.
//   warp 1      allocates 512 TMEM columns (one 128 x 320 fp32 accumulator);
//               lane 0 issues the tcgen05.mma and commits each tile.
//   warps 2..5  epilogue, one row per thread, 32 columns at a time: x_t from
//               TMEM, x_{t-1} from the lane above (a shuffle), from the
//               previous warp's last lane (a shared slot) or from x_prev at
//               t = 0; the taps in fp32 in the conv kernel's order; y stored as
//               bf16 (or fp32).
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace dflash2 {
namespace {

constexpr int kGcBN = 320;                                     // tile width (columns)
constexpr int kGcSubN = 160;                                   // per MMA / per TMA box
constexpr int kGcStages = 4;
constexpr int kGcThreads = 192;
constexpr int kGcABytes = 128 * kTileRowBytes;                 // 16 KB
constexpr int kGcBBytes = kGcBN * kTileRowBytes;               // 40 KB
constexpr int kGcStageBytes = kGcABytes + kGcBBytes;
constexpr uint32_t kGcTmemCols = 512;
constexpr uint32_t kGcIdesc = umma_idesc_bf16(128, kGcSubN);

struct GcSmem {
  uint64_t full[kGcStages];
  uint64_t empty[kGcStages];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
  float xch[2][4][32];     // last row of each epilogue warp, per 32-column chunk (double-buffered)
};

struct GcArgs {
  const uint16_t* x_prev;  // [B, d]
  const uint16_t* k0;      // [d]
  const uint16_t* k1;      // [d]
  const float* b_c;        // [2G] or null
  float* c;                // [M, 2G]
  unsigned int* ready;     // [m_tiles]: correction tiles stored per row tile
  void* y;                 // [M, d]
  int y_is_fp32;
  int M, L, d, K, R;       // R: rows per tile (whole blocks)
  int m_tiles, n_tiles;    // main tiles: m_tiles x n_tiles
  int c_tiles;             // correction tiles per row tile
};


// Named barrier `id` over `count` threads that also returns the AND of every
// thread's predicate, so the threads leave a loop together or not at all.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// tile -> (kind, row tile, column tile): the m_tiles * c_tiles correction tiles
// come first, then the main tiles row tile by row tile
struct GcTile {
  bool corr;
  int mt, nt;
};
__device__ __forceinline__ GcTile gc_tile(const GcArgs& a, int tile) {
  const int nc = a.m_tiles * a.c_tiles;
  if (tile < nc) return {true, tile / a.c_tiles, tile % a.c_tiles};
  tile -= nc;
  return {false, tile / a.n_tiles, tile % a.n_tiles};
}

__global__ void __launch_bounds__(kGcThreads, 1)
    gemm_conv_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmWc,
                     const GcArgs a, uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = align_smem<1024>(smem_raw);
  GcSmem& s = *reinterpret_cast<GcSmem*>(ring + kGcStages * kGcStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_all = a.m_tiles * (a.c_tiles + a.n_tiles);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGcStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.tfull, 1);
    mbar_init(&s.tempty, 4);            // one arrival per epilogue warp
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmWc);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem, kGcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();   // every operand tile is read by several CTAs
      int it = 0, issued = 0;
      for (int tile = blockIdx.x; tile < n_all && !*abort_flag; tile += gridDim.x) {
        const GcTile tl = gc_tile(a, tile);
        const int nk = (tl.corr ? a.d : a.K) / kBK;
        const CUtensorMap* ta = tl.corr ? &tmH : &tmA;
        const CUtensorMap* tb = tl.corr ? &tmWc : &tmW;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % kGcStages;
          if (it >= kGcStages && !mbar_wait_bounded(&s.empty[st], ((it / kGcStages) - 1) & 1, err)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* dst = ring + st * kGcStageBytes;
          mbar_arrive_expect_tx(&s.full[st], kGcStageBytes);
          tma_load_2d(dst, ta, kb * kBK, tl.mt * a.R, &s.full[st], pol);
          tma_load_2d(dst + kGcABytes, tb, kb * kBK, tl.nt * kGcBN, &s.full[st], pol);
          tma_load_2d(dst + kGcABytes + kGcSubN * kTileRowBytes, tb, kb * kBK, tl.nt * kGcBN + kGcSubN, &s.full[st],
                      pol);
          issued = it + 1;
        }
      }
      for (int j = issued - kGcStages > 0 ? issued - kGcStages : 0; j < issued; ++j)
        mbar_wait_bounded(&s.full[j % kGcStages], (j / kGcStages) & 1, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, i = 0;
      for (int tile = blockIdx.x; tile < n_all; tile += gridDim.x, ++i) {
        const GcTile tl = gc_tile(a, tile);
        const int nk = (tl.corr ? a.d : a.K) / kBK;
        if (i >= 1 && !mbar_wait_bounded(&s.tempty, (i - 1) & 1, err)) {   // the epilogue drained TMEM
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % kGcStages;
          if (!mbar_wait_bounded(&s.full[st], (it / kGcStages) & 1, err) || *abort_flag) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(ring + st * kGcStageBytes);
          const uint32_t b_base = a_base + kGcABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = umma_desc_sw128(a_base + k * 32);
            umma_bf16(tmem, ad, umma_desc_sw128(b_base + k * 32), kGcIdesc, (kb | k) != 0 ? 1u : 0u);
            umma_bf16(tmem + kGcSubN, ad, umma_desc_sw128(b_base + kGcSubN * kTileRowBytes + k * 32), kGcIdesc,
                      (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(&s.empty[st]);
        }
        umma_commit(&s.tfull);
        if (!ok) break;
      }
    }
  } else {
    // epilogue: thread = tile row r (TMEM lane); the q-th warp of the four owns lanes 32q..
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int G = a.d / 16, N = 2 * G;
    int i = 0, chunk = 0;
    for (int tile = blockIdx.x; tile < n_all; tile += gridDim.x, ++i) {
      const GcTile tl = gc_tile(a, tile);
      const int64_t m = static_cast<int64_t>(tl.mt) * a.R + r;
      const bool row_ok = r < a.R && m < a.M;
      bool ready = mbar_wait_bounded(&s.tfull, i & 1, err) && !*abort_flag;
      if (!tl.corr && threadIdx.x == 64 && ready) {
        // the row tile's corrections must all be stored before they are read
        const unsigned int* cnt = a.ready + tl.mt;
        if (ld_acquire(cnt) < static_cast<unsigned int>(a.c_tiles)) {
          const uint64_t t0 = global_timer_ns();
          for (uint32_t n = 1;; ++n) {
            if (ld_acquire(cnt) >= static_cast<unsigned int>(a.c_tiles)) break;
            if ((n & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
              raise_error(err, DFLASH2_DEVERR_TIMEOUT);
              ready = false;
              break;
            }
          }
        }
      }
      // the four warps meet at a named barrier per chunk: they decide together
      if (!named_bar_and(2, 128, ready)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const float* crow = a.c + m * N;
#pragma unroll 1
      for (int cc = 0; cc < kGcBN / 32; ++cc, ++chunk) {
        const int col0 = tl.nt * kGcBN + cc * 32;
        const bool live = row_ok && col0 < (tl.corr ? N : a.d);
        // this chunk's small operands first, so their latency hides behind the TMEM read
        uint4 k0v[4], k1v[4], xpv[4];
        float c0[2] = {0.f, 0.f}, c1[2] = {0.f, 0.f}, bias[32];
        const int t = static_cast<int>(m % a.L);
        if (!tl.corr && live) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            k0v[u] = reinterpret_cast<const uint4*>(a.k0 + col0)[u];
            k1v[u] = reinterpret_cast<const uint4*>(a.k1 + col0)[u];
          }
          const int g = col0 / 16;
          c0[0] = crow[g];
          c0[1] = crow[g + 1];
          c1[0] = crow[G + g];
          c1[1] = crow[G + g + 1];
          if (t == 0) {
            const uint4* xs = reinterpret_cast<const uint4*>(a.x_prev + (m / a.L) * a.d + col0);
#pragma unroll
            for (int u = 0; u < 4; ++u) xpv[u] = xs[u];
          }
        }
        if (tl.corr && live) {
#pragma unroll
          for (int j = 0; j < 32; ++j) bias[j] = (a.b_c && col0 + j < N) ? a.b_c[col0 + j] : 0.0f;
        }
        float v[32];
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + cc * 32, v);
        tmem_ld_wait();
        if (cc == kGcBN / 32 - 1) {
          // the accumulator is read out: the next tile's MMAs may start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.tempty);
        }
        if (tl.corr) {
          // c = acc + b_c; N is a multiple of 8, so columns come in whole groups of four
          if (live) {
            float* dst = a.c + m * N + col0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (col0 + j >= N) break;
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__fadd_rn(v[j], bias[j]), __fadd_rn(v[j + 1], bias[j + 1]),
                              __fadd_rn(v[j + 2], bias[j + 2]), __fadd_rn(v[j + 3], bias[j + 3]));
            }
          }
          continue;
        }
        // x_{t-1}: the lane above, or the previous warp's last lane through shared memory
        float* slot = s.xch[chunk & 1][q];
        if (lane == 31) {
#pragma unroll
          for (int j = 0; j < 32; ++j) slot[j] = v[j];
        }
        named_bar_sync(1, 128);
        float xp[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) xp[j] = __shfl_up_sync(0xFFFFFFFFu, v[j], 1);
        if (lane == 0 && q > 0) {
          const float* prev = s.xch[chunk & 1][q - 1];
#pragma unroll
          for (int j = 0; j < 32; ++j) xp[j] = prev[j];
        }
        if (!live) continue;
        if (t == 0) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t w[4] = {xpv[u].x, xpv[u].y, xpv[u].z, xpv[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xp[8 * u + 2 * e] = __uint_as_float(w[e] << 16);
              xp[8 * u + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
          }
        }
        float y[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w0[4] = {k0v[u].x, k0v[u].y, k0v[u].z, k0v[u].w};
          const uint32_t w1[4] = {k1v[u].x, k1v[u].y, k1v[u].z, k1v[u].w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = 8 * u + e;
            const uint32_t b0 = (e & 1) ? (w0[e >> 1] & 0xFFFF0000u) : (w0[e >> 1] << 16);
            const uint32_t b1 = (e & 1) ? (w1[e >> 1] & 0xFFFF0000u) : (w1[e >> 1] << 16);
            const float ka = __fadd_rn(__uint_as_float(b0), c0[j >> 4]);
            const float kb = __fadd_rn(__uint_as_float(b1), c1[j >> 4]);
            y[j] = __fmaf_rn(ka, v[j], __fmul_rn(kb, xp[j]));
          }
        }
        if (a.y_is_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.y) + m * a.d + col0);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
        } else {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(y[2 * j], y[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.y) + m * a.d + col0);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (tl.corr) {
        // every epilogue thread's stores are visible device-wide before the count rises
        __threadfence();
        named_bar_sync(3, 128);
        if (threadIdx.x == 64) atomicAdd(a.ready + tl.mt, 1u);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      umma_commit(&s.drain);
      mbar_wait_bounded(&s.drain, 0, err);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kGcTmemCols);
  }
}

}  // namespace

size_t gemm_conv_workspace_bytes(int64_t B, int64_t L, int64_t d) {
  // c, then one 4-byte counter per row tile (at most B * L of them), 16-byte aligned
  const size_t c_bytes = static_cast<size_t>(B * L) * static_cast<size_t>(2 * (d / 16)) * sizeof(float);
  return c_bytes + ((static_cast<size_t>(B * L) * sizeof(unsigned int) + 15) & ~size_t(15));
}

cudaError_t launch_gemm_conv2tap(const uint16_t* A, const uint16_t* W, const uint16_t* x_prev, const uint16_t* hs,
                                 const uint16_t* k0, const uint16_t* k1, const uint16_t* W_c, const float* b_c,
                                 int64_t B, int64_t L, int64_t K, int64_t d, float* c_work, void* y, int y_is_fp32,
                                 uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t M = B * L;
  if (K % kBK != 0 || d % 64 != 0 || L < 1 || L > 128 || M > 0x7FFFFFFF || K > 0x7FFFFFFF || d > 0x7FFFFFFF)
    return cudaErrorInvalidValue;
  const int64_t N = 2 * (d / 16);
  GcArgs ga;
  ga.x_prev = x_prev;
  ga.k0 = k0;
  ga.k1 = k1;
  ga.b_c = b_c;
  ga.c = c_work;
  ga.ready = reinterpret_cast<unsigned int*>(c_work + M * N);
  ga.y = y;
  ga.y_is_fp32 = y_is_fp32;
  ga.M = static_cast<int>(M);
  ga.L = static_cast<int>(L);
  ga.d = static_cast<int>(d);
  ga.K = static_cast<int>(K);
  ga.R = static_cast<int>((128 / L) * L);
  ga.m_tiles = static_cast<int>((M + ga.R - 1) / ga.R);
  ga.n_tiles = static_cast<int>((d + kGcBN - 1) / kGcBN);
  ga.c_tiles = static_cast<int>((N + kGcBN - 1) / kGcBN);
  const int64_t tiles = static_cast<int64_t>(ga.m_tiles) * (ga.n_tiles + ga.c_tiles);
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  CUtensorMap ta, tw, th, tc;
  if (!make_tmap_bf16_2d(&ta, A, M, K, K, 128) || !make_tmap_bf16_2d(&tw, W, d, K, K, kGcSubN) ||
      !make_tmap_bf16_2d(&th, hs, M, d, d, 128) || !make_tmap_bf16_2d(&tc, W_c, N, d, d, kGcSubN))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kGcStages * kGcStageBytes + sizeof(GcSmem);
  {
    const cudaError_t e = set_smem_limit<gemm_conv_kernel>(smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaMemsetAsync(ga.ready, 0, static_cast<size_t>(ga.m_tiles) * sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;
  // all CTAs resident (cooperative launch): a main tile's epilogue may wait for
  // a correction tile that another CTA computes
  const int grid = tiles < num_sms ? static_cast<int>(tiles) : num_sms;
  void* kargs[] = {&ta, &tw, &th, &tc, &ga, &err};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(gemm_conv_kernel), grid, kGcThreads, kargs, smem,
                                     stream);
}

}  // namespace dflash2
