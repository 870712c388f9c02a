// proj.cu -- the path selector in projection form ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector"): the 256-dimensional embeddings of
// the score equation are projections of the shared token embedding,
//   A(a) = W_A E(a),   B(b) = W_B E(b),
// computed on the fly for exactly the tokens a step needs instead of being
// read from [V, 256] tables.
//
// proj_kernel (persistent, one CTA per SM) computes, on the tensor cores,
//   P[m, 0:256]   = W_A E(id_m),   P[m, 256:512] = W_B E(id_m)      (fp32)
// for the rows m of the step: the B*L*16 candidates (row (b*L + t)*16 + j),
// then the B last verified tokens.  Tiles are 128 rows x 256 columns (one of
// W_A / W_B); consecutive tiles share their rows, so the second read of each
// gathered row hits L2.  A 4-deep ring of 48 KB stages (64-wide K blocks):
//   warps 6..9  gather the tile's 128 embedding rows with 16-byte cp.async
//               (8 lanes per row, so each instruction reads 4 whole 128-byte
//               row segments) straight into the 128-byte-swizzled K-major
//               layout; each thread waits for its copies two stages later,
//               makes them visible to the tensor cores (fence.proxy.async)
//               and arrives on the stage's barrier.  TMA tile::gather4 does
//               the same job but issues one row at a time and capped the
//               kernel at a fifth of the tensor rate.
//   warp 0      lane 0 loads the 256 x 64 W tile of each stage with TMA.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators);
//               lane 0 issues the tcgen05.mma and commits each finished tile.
//   warps 2..5  epilogue: one row per thread, tcgen05.ld 32 columns at a time,
//               16-byte stores into P; overlaps the next tile's MMAs.
// pair_proj_kernel: one CTA per block position, as the table-form pair kernel
// but reading the predecessors' A rows and the candidates' B rows from P
// (fp32, contiguous per position) instead of gathering table rows.
#include "common.cuh"
#include "launch.h"
#include "pair_math.cuh"
#include "tcgen05.cuh"

namespace dflash2 {
namespace {

constexpr int kPjBN = kEmbed;
constexpr int kPjStages = 4;
constexpr int kPjThreads = 320;                                // 10 warps
constexpr int kPjGatherWarp0 = 6;                              // warps 6..9 gather A
constexpr int kPjGatherThreads = 128;
constexpr int kPjLag = 2;                                      // stages a gather thread keeps in flight
constexpr int kPjABytes = 128 * kTileRowBytes;                 // 16 KB
constexpr int kPjBBytes = kPjBN * kTileRowBytes;               // 32 KB
constexpr int kPjStageBytes = kPjABytes + kPjBBytes;
constexpr uint32_t kPjTmemCols = 2 * kPjBN;                    // double-buffered accumulator
constexpr uint32_t kPjIdesc = umma_idesc_bf16(128, kPjBN);
constexpr int kPjRowFloats = 2 * kEmbed;                       // P row: A then B

struct PjSmem {
  uint64_t full[kPjStages];
  uint64_t empty[kPjStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

// 16-byte asynchronous copy global -> shared (L2 only), completion tracked
// per thread by commit / wait groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (the tensor cores' operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Token of projection row m: a candidate (m < n_cand) or a last verified token;
// rows past the end gather token 0 (their results are not stored).
__device__ __forceinline__ int32_t proj_row_token(const int32_t* __restrict__ cand_idx,
                                                  const int32_t* __restrict__ last_verified, int64_t m,
                                                  int64_t n_cand, int64_t n_rows, int64_t V, uint32_t* err) {
  if (m >= n_rows) return 0;
  return clamp_token(m < n_cand ? cand_idx[m] : last_verified[m - n_cand], V, err);
}

__global__ void __launch_bounds__(kPjThreads, 1)
    proj_kernel(const uint16_t* __restrict__ E, const __grid_constant__ CUtensorMap tmWA,
                const __grid_constant__ CUtensorMap tmWB, const int32_t* __restrict__ cand_idx,
                const int32_t* __restrict__ last_verified, int64_t n_cand, int64_t n_rows, int64_t V, int d,
                int n_tiles, float* __restrict__ P, uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = align_smem<1024>(smem_raw);
  PjSmem& s = *reinterpret_cast<PjSmem*>(ring + kPjStages * kPjStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = d / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPjStages; ++i) {
      mbar_init(&s.full[i], kPjGatherThreads + 1);   // every gather thread + the W load
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], 4);       // one arrival per epilogue warp
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmWA);
    tma_prefetch_desc(&tmWB);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem, kPjTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      uint64_t pol_w;                                 // W_A, W_B: re-read by every tile
      asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_w));
      int it = 0, issued = 0;
      for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % kPjStages;
          if (it >= kPjStages && !mbar_wait_bounded(&s.empty[st], ((it / kPjStages) - 1) & 1, err)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&s.full[st], kPjBBytes);
          tma_load_2d(ring + st * kPjStageBytes + kPjABytes, (tile & 1) ? &tmWB : &tmWA, kb * kBK, 0, &s.full[st],
                      pol_w);
          issued = it + 1;
        }
      }
      // no TMA copy into the ring may still be in flight when the CTA exits
      for (int j = issued - kPjStages > 0 ? issued - kPjStages : 0; j < issued; ++j)
        mbar_wait_bounded(&s.full[j % kPjStages], (j / kPjStages) & 1, err);
    }
  } else if (warp >= kPjGatherWarp0) {
    // gather thread g: 16-byte chunk c = g % 8 of rows g / 8 + 16 i (i < 8)
    const int g = threadIdx.x - kPjGatherWarp0 * 32;
    const int c = g & 7, r0 = g >> 3;
    int it = 0, announced = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const int64_t m0 = static_cast<int64_t>(tile >> 1) * 128;
      const uint16_t* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        src[i] = E + static_cast<int64_t>(proj_row_token(cand_idx, last_verified, m0 + r0 + 16 * i, n_cand, n_rows,
                                                         V, err)) * d + c * 8;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int st = it % kPjStages;
        if ((it >= kPjStages && !mbar_wait_bounded(&s.empty[st], ((it / kPjStages) - 1) & 1, err)) || *abort_flag) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        uint8_t* a_st = ring + st * kPjStageBytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = r0 + 16 * i;                 // row & 7 == r0 & 7
          cp_async16(a_st + row * kTileRowBytes + ((c ^ (row & 7)) << 4), src[i] + kb * kBK);
        }
        cp_async_commit();
        if (it >= kPjLag) {
          cp_async_wait<kPjLag>();
          fence_proxy_async_smem();
          mbar_arrive(&s.full[(it - kPjLag) % kPjStages]);
          announced = it - kPjLag + 1;
        }
      }
    }
    // the last stages: wait for every copy, then announce them
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int j = announced; j < it; ++j) mbar_arrive(&s.full[j % kPjStages]);
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, i = 0;
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait_bounded(&s.tempty[buf], ((i >> 1) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * kPjBN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % kPjStages;
          if (!mbar_wait_bounded(&s.full[st], (it / kPjStages) & 1, err) || *abort_flag) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(ring + st * kPjStageBytes);
          const uint32_t b_base = a_base + kPjABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16(acc, umma_desc_sw128(a_base + k * 32), umma_desc_sw128(b_base + k * 32), kPjIdesc,
                      (kb | k) != 0 ? 1u : 0u);
          umma_commit(&s.empty[st]);
        }
        umma_commit(&s.tfull[buf]);
        if (!ok) break;
      }
    }
  } else {
    // epilogue: one projection row per thread
    const int q = warp & 3;
    int i = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++i) {
      const int buf = i & 1;
      if (!mbar_wait_bounded(&s.tfull[buf], (i >> 1) & 1, err) || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(tile >> 1) * 128 + q * 32 + lane;
      float* dst = P + row * kPjRowFloats + (tile & 1) * kPjBN;
#pragma unroll 1
      for (int c = 0; c < kPjBN / 32; ++c) {
        float v[32];
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kPjBN + c * 32, v);
        tmem_ld_wait();
        if (row < n_rows) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[buf]);
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
    tmem_dealloc(tmem, kPjTmemCols);
  }
}

// One CTA per block position (b, t): G = A(pred_i) (.) H_t and Bc = B(cand_j)
// from P, then the 16 x 16 products.
__global__ void __launch_bounds__(256) pair_proj_kernel(const float* __restrict__ cand_val,
                                                        const float* __restrict__ gate, const float* __restrict__ P,
                                                        int64_t L, int64_t n_cand, float* __restrict__ S) {
  __shared__ __align__(16) float G[kTopK][kEmbed];
  __shared__ __align__(16) float Bc[kTopK][kEmbed];
  const int tid = threadIdx.x;
  const int64_t pos = blockIdx.x;              // b * L + t
  const int64_t b = pos / L, t = pos % L;
  const float* Ht = gate + pos * kEmbed;
  // 32 rows x 64 float4 = 2048 loads, 8 per thread, all issued before any use
  constexpr int kPer = 2 * kTopK * (kEmbed / 4) / 256;
  float4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * 256;
    const int row = e / (kEmbed / 4), ch = e % (kEmbed / 4);
    const int r16 = row & (kTopK - 1);
    const int64_t src = row < kTopK ? ((t == 0 ? n_cand + b : (pos - 1) * kTopK + r16) * kPjRowFloats)
                                    : ((pos * kTopK + r16) * kPjRowFloats + kEmbed);
    v[u] = *reinterpret_cast<const float4*>(P + src + ch * 4);
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid + u * 256;
    const int row = e / (kEmbed / 4), ch = e % (kEmbed / 4);
    const int r16 = row & (kTopK - 1);
    if (row < kTopK) {
      const float4 h = *reinterpret_cast<const float4*>(Ht + ch * 4);
      *reinterpret_cast<float4*>(&G[r16][ch * 4]) =
          make_float4(__fmul_rn(v[u].x, h.x), __fmul_rn(v[u].y, h.y), __fmul_rn(v[u].z, h.z), __fmul_rn(v[u].w, h.w));
    } else {
      *reinterpret_cast<float4*>(&Bc[r16][ch * 4]) = v[u];
    }
  }
  __syncthreads();
  pair_products(G, Bc, cand_val, S, pos, tid);
}

}  // namespace

size_t proj_rows(int64_t B, int64_t L) { return static_cast<size_t>(B * L * kTopK + B); }

size_t proj_workspace_bytes(int64_t B, int64_t L) {
  return proj_rows(B, L) * kPjRowFloats * sizeof(float);
}

cudaError_t launch_pair_scores_proj(const int32_t* cand_idx, const float* cand_val, const int32_t* last_verified,
                                    const float* gate, const uint16_t* E, const uint16_t* W_A, const uint16_t* W_B,
                                    int64_t B, int64_t L, int64_t d, int64_t V, float* P, float* S, int num_sms,
                                    uint32_t* err, cudaStream_t stream) {
  if (d % kBK != 0 || d > 0x7FFFFFFF || V > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int64_t n_cand = B * L * kTopK;
  const int64_t n_rows = static_cast<int64_t>(proj_rows(B, L));
  const int64_t m_tiles = (n_rows + 127) / 128;
  if (2 * m_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const int n_tiles = static_cast<int>(2 * m_tiles);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, W_A, kEmbed, d, d, kPjBN) ||
      !make_tmap_bf16_2d(&tb, W_B, kEmbed, d, d, kPjBN))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kPjStages * kPjStageBytes + sizeof(PjSmem);
  {
    const cudaError_t e = set_smem_limit<proj_kernel>(smem);
    if (e != cudaSuccess) return e;
  }
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  proj_kernel<<<grid, kPjThreads, smem, stream>>>(E, ta, tb, cand_idx, last_verified, n_cand, n_rows, V,
                                                  static_cast<int>(d), n_tiles, P, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pair_proj_kernel<<<static_cast<unsigned>(B * L), 256, 0, stream>>>(cand_val, gate, P, L, n_cand, S);
  return cudaGetLastError();
}

}  // namespace dflash2
