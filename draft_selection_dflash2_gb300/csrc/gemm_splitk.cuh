// gemm_splitk.cuh -- tcgen05 GEMM split over K across a thread-block cluster,
// reduced through distributed shared memory, with a pluggable epilogue.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]      A: [M, K] bf16, B: [N, K] bf16, fp32 accumulate
//
// Grid (ks, n_tiles, m_tiles) with clusters of (ks, 1, 1): the ks CTAs of a
// cluster own the same 128 x BN output tile and split its K loop.  Each CTA:
//   warp 0        TMA producer: 128 x 64 A tiles and BN x 64 B tiles (B may be
//                 assembled from several boxes, Epi::load_b) into a ring of
//                 `stages` slots.
//   warp 1        allocates TMEM; lane 0 issues the stage's tcgen05.mma: BN is
//                 covered by `Epi::sub_n`-wide instructions (BN > 256 needs two),
//                 then commits the stage back to the producer.
//   warps 6..11   idle until the epilogue, which all twelve warps share.
//   warps 2..5    read the finished fp32 partial from TMEM (tcgen05.ld), turn each
//                 32 x 32 block around in a small shared buffer, and push whole
//                 row segments, as 16-byte stores through distributed shared
//                 memory, into the CTA of the cluster that owns those rows: rank r
//                 owns rows [r * 128/ks, (r + 1) * 128/ks) and keeps one slot per
//                 source rank.  A first cluster barrier, entered by every warp once
//                 its part of the K loop is over, guarantees that no peer still
//                 loads into or multiplies out of the ring the slots overwrite.
// After a second cluster barrier every rank holds all ks partials of its own
// rows in local shared memory, and all 384 threads run Epi::finish on them
// (which may reuse the rest of the region, e.g. to stage its own inputs).
// Every mbarrier wait is bounded (DFLASH2_DEVERR_TIMEOUT, then drain and exit).
#pragma once

#include <cooperative_groups.h>

#include "launch.h"
#include "tcgen05.cuh"

namespace dflash2 {

constexpr int kSkThreads = 384;
constexpr int kSkMaxStages = 6;
constexpr int kSkCtrlBytes = 256;
constexpr int kSkMaxSmem = 232448;                   // 227 KB: the opt-in per-block limit
constexpr int kSkXposePitch = 36;                    // floats per row of a warp's 32 x 32 buffer
constexpr int kSkXposeBytes = 2 * 4 * 32 * kSkXposePitch * 4;   // two per epilogue warp

struct SplitKShape {
  int M, K, BN;          // BN: tile width in output columns (multiple of 32)
  int ks;                // cluster size = number of K splits
  int n_tiles, m_tiles;
  uint32_t tmem_cols;    // power of two >= BN
  int stages;            // ring depth (sk_plan)
  int region_bytes;      // ring / slot region at the 1024-aligned base (sk_plan)
};

__host__ __device__ inline int sk_stage_bytes(int BN) { return 128 * kTileRowBytes + BN * kTileRowBytes; }
// fp32 words per slot row: 16-byte aligned rows; a pitch of 4 (mod 32) words
// keeps 8 consecutive rows' float4 accesses on distinct banks
__host__ __device__ inline int sk_partial_pitch(int BN) { return BN + 4; }
__host__ __device__ inline int sk_slots_bytes(int BN) { return 128 * sk_partial_pitch(BN) * 4; }

// Picks the ring depth (as deep as fits, up to kSkMaxStages) and the size of
// the region that holds the ring during the K loop and the slots plus the
// transpose buffers after it.  False if not even two stages fit.
__host__ inline bool sk_plan(SplitKShape& sh) {
  const int need = sk_slots_bytes(sh.BN) + kSkXposeBytes;
  for (int s = kSkMaxStages; s >= 2; --s) {
    const int ring = s * sk_stage_bytes(sh.BN);
    const int region = ring > need ? ring : need;
    if (1024 + region + kSkCtrlBytes <= kSkMaxSmem) {
      sh.stages = s;
      sh.region_bytes = region;
      return true;
    }
  }
  return false;
}
__host__ inline size_t sk_smem_bytes(const SplitKShape& sh) {
  return 1024 + static_cast<size_t>(sh.region_bytes) + kSkCtrlBytes;
}

// Picks the cluster size: the largest power of two <= 8 that keeps the grid
// within one wave of the SMs and leaves every CTA at least two K blocks.
__host__ inline int sk_choose_ks(int tiles, int nk, int num_sms) {
  int ks = 1;
  while (ks < 8 && tiles * ks * 2 <= num_sms && nk >= ks * 4) ks *= 2;
  return ks;
}

// The ks partial slots of this rank's rows, in local shared memory: slot q
// holds source rank q's partial of local rows [0, 128/ks).
struct SkPartials {
  const float* base;
  int ks, pitch, rows_per;

  __device__ SkPartials(const float* slots, int ks_, int pitch_)
      : base(slots), ks(ks_), pitch(pitch_), rows_per(128 / ks_) {}

  template <int KS>
  __device__ __forceinline__ float4 sum4_k(int lr, int col) const {
    float4 v[KS];
#pragma unroll
    for (int q = 0; q < KS; ++q) v[q] = *reinterpret_cast<const float4*>(base + (q * rows_per + lr) * pitch + col);
    float4 a = v[0];
#pragma unroll
    for (int q = 1; q < KS; ++q) {
      a.x += v[q].x;
      a.y += v[q].y;
      a.z += v[q].z;
      a.w += v[q].w;
    }
    return a;
  }

  // Sum over the source ranks of columns [col, col + 4) (col % 4 == 0) of local
  // row `lr`: every slot's load is issued before any add, and the adds run in
  // rank order, so the result does not depend on timing.
  __device__ __forceinline__ float4 sum4(int lr, int col) const {
    switch (ks) {
      case 1: return sum4_k<1>(lr, col);
      case 2: return sum4_k<2>(lr, col);
      case 4: return sum4_k<4>(lr, col);
      default: return sum4_k<8>(lr, col);
    }
  }
};

template <class Epi>
__global__ void __launch_bounds__(kSkThreads, 1)
    splitk_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const SplitKShape sh, const typename Epi::Params p, uint32_t* __restrict__ err) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  const int stage_bytes = sk_stage_bytes(sh.BN);
  const int S = sh.stages;
  uint8_t* ctrl = smem + sh.region_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kSkMaxStages;
  uint64_t* acc_bar = empty + kSkMaxStages;
  uint64_t* drain_bar = acc_bar + 1;
  uint64_t* epi_bars = drain_bar + 1;                        // two, for Epi::finish
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* slots = reinterpret_cast<float*>(smem);             // reuses the ring after the K loop
  float* xpose = reinterpret_cast<float*>(smem + sk_slots_bytes(sh.BN));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster.block_rank());
  const int n_tile = blockIdx.y, m_tile = blockIdx.z;
  const int m0 = m_tile * 128;
  const int nk = sh.K / kBK;
  const int kb0 = static_cast<int>((static_cast<int64_t>(nk) * rank) / sh.ks);
  const int kb1 = static_cast<int>((static_cast<int64_t>(nk) * (rank + 1)) / sh.ks);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(&epi_bars[0], 1);
    mbar_init(&epi_bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, sh.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait_bounded(&empty[s], ((i / S) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        uint8_t* a_dst = smem + s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d(a_dst, &tmA, (kb0 + i) * kBK, m0, &full[s], pol);
        Epi::load_b(a_dst + 128 * kTileRowBytes, &tmB, (kb0 + i) * kBK, n_tile, p, &full[s], pol);
        issued = i + 1;
      }
      for (int i = issued - S > 0 ? issued - S : 0; i < issued; ++i) mbar_wait_bounded(&full[i % S], (i / S) & 1, err);
    }
    __syncwarp();
    cluster_arrive();   // no TMA write into this CTA's ring is outstanding
    cluster_wait();
  } else if (warp == 1) {
    if (lane == 0) {
      const int sub_n = Epi::sub_n(sh.BN);
      const uint32_t idesc = umma_idesc_bf16(128, sub_n);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % S;
        if (!mbar_wait_bounded(&full[s], (i / S) & 1, err) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_addr(smem + s * stage_bytes);
        const uint32_t b_base = a_base + 128 * kTileRowBytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          for (int n0 = 0; n0 < sh.BN; n0 += sub_n)
            umma_bf16(tmem + n0, umma_desc_sw128(a_base + k * 32),
                      umma_desc_sw128(b_base + n0 * kTileRowBytes + k * 32), idesc, (i | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_bar);
    }
    __syncwarp();
    cluster_arrive();   // the epilogue warps' arrivals vouch for the MMAs' completion
    cluster_wait();
  } else if (warp >= 6) {
    cluster_arrive();
    cluster_wait();
  } else {
    // Warp q (= warp & 3) may read TMEM lanes [32q, 32q + 32): tile rows 32q.. .
    const int q = warp & 3;
    const int rows_per = 128 / sh.ks;
    const int pitch = sk_partial_pitch(sh.BN);
    const bool ok = mbar_wait_bounded(acc_bar, 0, err) && !*abort_flag;
    cluster_arrive();   // every CTA of the cluster has seen its own MMAs complete:
    cluster_wait();     // no peer reads or loads its ring any more
    tc_fence_after();
    // this lane stores columns [(lane % 8) * 4, +4) of rows 32q + 4i + lane / 8 (i < 8)
    float* dst[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = q * 32 + i * 4 + (lane >> 3);
      dst[i] = cluster.map_shared_rank(slots, row / rows_per) + (rank * rows_per + row % rows_per) * pitch +
               (lane & 7) * 4;
    }
    float* xp = xpose + q * 2 * 32 * kSkXposePitch;
    const bool keep = ok && nkb > 0;
    const int nc = sh.BN / 32;
    // two 32-column chunks per step: both TMEM loads, then both turns, then 16 stores in flight
    for (int c = 0; c < nc; c += 2) {
      const int nb = c + 1 < nc ? 2 : 1;
      float v[2][32];
#pragma unroll
      for (int b = 0; b < 2; ++b)
        if (b < nb) tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + (c + b) * 32, v[b]);
      tmem_ld_wait();
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        if (b >= nb) break;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(xp + (b * 32 + lane) * kSkXposePitch + j) =
              keep ? make_float4(v[b][j], v[b][j + 1], v[b][j + 2], v[b][j + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncwarp();
      float4 t[2][8];
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (b < nb)
            t[b][i] = *reinterpret_cast<const float4*>(xp + (b * 32 + i * 4 + (lane >> 3)) * kSkXposePitch +
                                                       (lane & 7) * 4);
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (b < nb) *reinterpret_cast<float4*>(dst[i] + (c + b) * 32) = t[b][i];
      __syncwarp();
    }
    tc_fence_before();
  }
  cluster_arrive();   // this CTA's pushes are complete ...
  cluster_wait();     // ... and so are every peer's into this CTA
  if (!*abort_flag) Epi::finish(p, sh, smem, epi_bars, m0, n_tile, rank, threadIdx.x, err);
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, err);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, sh.tmem_cols);
  }
}

template <class Epi>
cudaError_t launch_splitk_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const SplitKShape& sh,
                               const typename Epi::Params& p, uint32_t* err, cudaStream_t stream) {
  const size_t smem = sk_smem_bytes(sh);
  {
    const cudaError_t e = set_smem_limit<splitk_gemm_kernel<Epi>>(smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sh.ks, sh.n_tiles, sh.m_tiles);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = sh.ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, splitk_gemm_kernel<Epi>, tmA, tmB, sh, p, err);
}

}  // namespace dflash2
