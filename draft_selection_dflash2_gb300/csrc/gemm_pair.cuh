// gemm_pair.cuh -- tcgen05 GEMM over CTA pairs, split over K, writing fp32
// partial sums to global memory.
//
//   P[q][m, n] = sum_{k in split q} A[m, k] * B[n, k]
//   A: [M, K] bf16 (K-major), B: [N, K] bf16 (K-major), fp32 accumulate.
//
// A CTA pair (a cluster of 2) computes a 256 x BN tile with
// tcgen05.mma.cta_group::2: each CTA holds its own 128 rows of A and half of
// every B sub-block, so one 64-wide K stage brings 128 + BN/2 rows (36 KB at
// BN = 320) into each SM instead of 128 + BN: what an SM can take in per clock
// bounds these GEMMs, and the pair cuts it by a third.  The K loop is split
// over ks pairs that work independently and store their fp32 partials to
// P[q] (the consumer sums the ks partials in a fixed order, so the result does
// not depend on timing); no cluster reduction or barrier is needed beyond the
// pair.
// Grid (2 ks, n_tiles, m_pairs), clusters of (2, 1, 1); rank 0 of a pair leads.
//   warp 0       TMA producer: this CTA's 128 x 64 A tile and its half of each
//                B sub-block into a ring; both CTAs' copies complete on the
//                leader's stage barrier.
//   warp 1       allocates TMEM (cta_group::2); the leader's lane 0 issues the
//                pair MMAs (one per B sub-block and 16-wide K step) and commits
//                each stage back to both producers.
//   warps 2..5   epilogue: each thread owns one row (TMEM lane); per 32
//                columns (tcgen05.ld) the warp's 32 x 32 block goes to shared
//                memory in the 128-byte-swizzled layout (a thread's eight
//                16-byte pieces land on distinct bank groups) and leaves by one
//                TMA tensor store, double-buffered per warp.  Blocks that are
//                only partly valid (ragged shapes) are stored by guarded float4
//                writes instead.
// The B tile is Shape::kSubs sub-blocks of BN / kSubs columns; CTA rank holds
// BN / kSubs / 2 of each sub-block's rows, from B row Shape::b_row(t, s, rank,
// BN / kSubs / 2) on (sub-block s of n-tile t), and the pair MMA takes rank 0's
// rows as the sub-block's first columns; tile columns [c, c + 4) (c % 4 == 0) go to output columns
// Shape::out_col(t, c) + [0, 4) (or nowhere when Shape::valid(t, c) is false).
// Every mbarrier wait is bounded (DFLASH2_DEVERR_TIMEOUT, then drain and exit).
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace dflash2 {

constexpr int kPgThreads = 192;
constexpr int kPgMaxStages = 8;
constexpr int kPgABytes = 128 * kTileRowBytes;   // 16 KB
constexpr int kPgMaxSmem = 232448;               // 227 KB: the opt-in per-block limit

struct PairGemmShape {
  int M, K, N;      // N: the partials' row length (output columns)
  int BN;           // tile width (multiple of 32, <= 512)
  int ks;           // K splits
  int n_tiles, m_pairs;
  int stages;
  uint32_t tmem_cols;   // power of two >= BN
};

__host__ __device__ inline int pg_stage_bytes(int BN) { return kPgABytes + (BN / 2) * kTileRowBytes; }

struct PgSmem {
  uint64_t full[kPgMaxStages];    // the leader's count both CTAs' bytes
  uint64_t empty[kPgMaxStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

__host__ inline size_t pg_smem_bytes(const PairGemmShape& sh) {
  return 1024 + static_cast<size_t>(sh.stages) * pg_stage_bytes(sh.BN) + sizeof(PgSmem);
}

// Ring depth: as deep as fits (at most kPgMaxStages); false if not two.
__host__ inline bool pg_plan(PairGemmShape& sh) {
  for (int s = kPgMaxStages; s >= 2; --s) {
    sh.stages = s;
    if (pg_smem_bytes(sh) <= static_cast<size_t>(kPgMaxSmem)) return true;
  }
  return false;
}

__device__ __forceinline__ uint32_t pg_cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t pg_cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// The box at (x, y) into this CTA's shared memory, completing tx bytes on the
// barrier at cluster address `bar` (the leader's).
__device__ __forceinline__ void pg_tma_load(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// D[tmem] (+)= A B^T over both CTAs' operands at the same shared offsets.
__device__ __forceinline__ void pg_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` in both CTAs when the pair's MMAs so far are complete.
__device__ __forceinline__ void pg_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Arrives once on this CTA's `bar` when the pair's MMAs so far are complete.
__device__ __forceinline__ void pg_commit_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// A 32 x 32 fp32 block from shared memory to the box at (x, y, z) of a 3-D
// tensor map, in the current bulk group.
__device__ __forceinline__ void pg_tma_store(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
      : "memory");
}

template <class Shape>
__global__ void __launch_bounds__(kPgThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmP, const PairGemmShape sh,
                     const typename Shape::Params sp, float* __restrict__ part, uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = align_smem<1024>(smem_raw);
  const int stage_bytes = pg_stage_bytes(sh.BN);
  const int S = sh.stages;
  PgSmem& s = *reinterpret_cast<PgSmem*>(ring + S * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = pg_cluster_rank();
  const bool leader = rank == 0;
  const int q = blockIdx.x >> 1, n_tile = blockIdx.y, m_pair = blockIdx.z;
  const int m0 = m_pair * 256 + static_cast<int>(rank) * 128;   // this CTA's rows
  const int nk = sh.K / kBK;
  const int kb0 = static_cast<int>((static_cast<int64_t>(nk) * q) / sh.ks);
  const int kb1 = static_cast<int>((static_cast<int64_t>(nk) * (q + 1)) / sh.ks);
  const int sub_n = sh.BN / Shape::kSubs;   // columns per MMA
  const int half = sub_n / 2;               // B rows per CTA per sub-block

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.tfull, 1);
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s.tmem)),
                 "r"(sh.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers and TMEM exist before any remote arrival or pair MMA
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  volatile int* abort_flag = &s.abort_flag;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_last();   // A rows: read by every n-tile
      const uint64_t pol_b = l2_policy_evict_last();   // B rows: read by every row pair
      const uint32_t bar0 = pg_cluster_addr(&s.full[0], 0);
      int issued = 0;
      for (int i = 0; i < kb1 - kb0 && !*abort_flag; ++i) {
        const int st = i % S;
        if (i >= S && !mbar_wait_bounded(&s.empty[st], ((i / S) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        uint8_t* a_dst = ring + st * stage_bytes;
        if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * stage_bytes);
        const uint32_t bar = bar0 + static_cast<uint32_t>(st) * 8u;
        const int kx = (kb0 + i) * kBK;
        pg_tma_load(a_dst, &tmA, kx, m0, bar, pol_a);
        for (int sb = 0; sb < Shape::kSubs; ++sb)
          pg_tma_load(a_dst + kPgABytes + sb * half * kTileRowBytes, &tmB, kx,
                      Shape::b_row(sp, n_tile, sb, static_cast<int>(rank), half), bar, pol_b);
        issued = i + 1;
      }
      // before this CTA may exit: its own copies have landed (the leader's
      // barrier saw them) and the pair's MMAs are done with every stage
      for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j) {
        if (leader) mbar_wait_bounded(&s.full[j % S], (j / S) & 1, err);
        mbar_wait_bounded(&s.empty[j % S], (j / S) & 1, err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t idesc = umma_idesc_bf16(256, sub_n);
      for (int i = 0; i < kb1 - kb0; ++i) {
        const int st = i % S;
        if (!mbar_wait_bounded(&s.full[st], (i / S) & 1, err) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_addr(ring + st * stage_bytes);
        const uint32_t b_base = a_base + kPgABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t ad = umma_desc_sw128(a_base + k * 32);
          for (int sb = 0; sb < Shape::kSubs; ++sb)
            pg_mma(tmem + sb * sub_n, ad, umma_desc_sw128(b_base + sb * half * kTileRowBytes + k * 32), idesc,
                   (i | k) != 0 ? 1u : 0u);
        }
        pg_commit_both(&s.empty[st]);
      }
      pg_commit_both(&s.tfull);
    }
  } else {
    // epilogue: warp w reads TMEM lanes [32 (w & 3), +32): one row per thread
    const int wq = warp & 3;
    const int row = m0 + wq * 32 + lane;
    const bool ok = mbar_wait_bounded(&s.tfull, 0, err) && !*abort_flag;
    tc_fence_after();
    float* dst = part + (static_cast<int64_t>(q) * sh.M + row) * sh.N;
    const bool empty_split = kb1 <= kb0;
    // the ring is free once the MMAs are complete: two 4 KB staging blocks per warp
    uint8_t* stage = ring + wq * 2 * 4096;
#pragma unroll 1
    for (int c = 0, i = 0; c < sh.BN; c += 32, ++i) {
      float v[32];
      tmem_ld_x32(tmem + (static_cast<uint32_t>(wq * 32) << 16) + c, v);
      tmem_ld_wait();
      if (empty_split) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.0f;
      }
      if (!ok) continue;
      if (Shape::valid(sp, n_tile, c + 28) && Shape::out_col(sp, n_tile, c + 28) == Shape::out_col(sp, n_tile, c) + 28) {
        // the whole block is valid and contiguous: one TMA store (rows past M clip in the map)
        uint8_t* buf = stage + (i & 1) * 4096;
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // this buffer's last store
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          pg_tma_store(&tmP, buf, Shape::out_col(sp, n_tile, c), m0 + wq * 32, q);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      } else if (row < sh.M) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (Shape::valid(sp, n_tile, c + j))
            *reinterpret_cast<float4*>(dst + Shape::out_col(sp, n_tile, c + j)) =
                make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      }
    }
    // the stores are complete (and no longer read shared memory) before the CTA moves on
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1 && leader) {
    if (lane == 0) {
      pg_commit_local(&s.drain);
      mbar_wait_bounded(&s.drain, 0, err);
    }
    __syncwarp();
  }
  // the leader's MMAs are complete and every remote arrival has landed before
  // either CTA frees its TMEM or leaves
  tc_fence_before();
  cluster_arrive();
  cluster_wait();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(sh.tmem_cols) : "memory");
  }
}

template <class Shape>
cudaError_t launch_pair_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const PairGemmShape& sh,
                             const typename Shape::Params& sp, float* part, uint32_t* err, cudaStream_t stream) {
  CUtensorMap tmP;
  if (!make_tmap_f32_3d(&tmP, part, static_cast<uint64_t>(sh.N), static_cast<uint64_t>(sh.M),
                        static_cast<uint64_t>(sh.ks), 32, 32))
    return cudaErrorInvalidValue;
  const size_t smem = pg_smem_bytes(sh);
  {
    const cudaError_t e = set_smem_limit<pair_gemm_kernel<Shape>>(smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * sh.ks, sh.n_tiles, sh.m_pairs);
  cfg.blockDim = dim3(kPgThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<Shape>, tmA, tmB, tmP, sh, sp, part, err);
}

// K splits for a grid of `pairs` pair tiles: the largest (at most 8) that
// keeps 2 * pairs * ks CTAs within the resident slots and leaves each split at
// least 4 K blocks.
__host__ inline int pg_choose_ks(int pairs, int nk, int slots) {
  int ks = 1;
  while (ks < 8 && 2 * pairs * (ks + 1) <= slots && nk >= 4 * (ks + 1)) ++ks;
  return ks;
}

}  // namespace dflash2
