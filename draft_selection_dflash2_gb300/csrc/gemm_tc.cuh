// gemm_tc.cuh -- warp-specialised tcgen05 GEMM with a pluggable epilogue.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]      A: [M, K] bf16, B: [N, K] bf16, fp32 accumulate
//
// One CTA computes one 128 x BN output tile over the whole K:
//   warp 0        TMA producer: streams 128 x 64 A tiles and BN x 64 B tiles
//                 (128-byte swizzle) into a STAGES-deep shared-memory ring.
//   warp 1        allocates BN TMEM columns; lane 0 issues 4 tcgen05.mma
//                 (128 x BN x 16) per stage and commits the stage back to the
//                 producer, then commits the finished accumulator.
//   warps 2..5    epilogue: tcgen05.ld of the accumulator, 32 columns at a time
//                 (warp w reads TMEM lanes 32 (w % 4) .. +31 = its 32 rows), fed
//                 to Epi::consume.  Epi::finish then runs on all 192 threads.
// Every mbarrier wait is bounded; a timeout raises DFLASH2_DEVERR_TIMEOUT and the
// CTA drains its in-flight copies and MMAs before freeing TMEM and exiting.
#pragma once

#include "tcgen05.cuh"

namespace dflash2 {

constexpr int kGemmThreads = 192;

template <int BN, int STAGES>
struct GemmLayout {
  static constexpr int kABytes = 128 * kTileRowBytes;     // 16 KB
  static constexpr int kBBytes = BN * kTileRowBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  // full[STAGES], empty[STAGES], acc, drain, tmem address, abort flag, consumed count
  static constexpr int kBarBytes = (2 * STAGES + 2) * 8 + 16;
  static constexpr int kEpiOffset = (kBarOffset + kBarBytes + 127) / 128 * 128;
  static constexpr uint32_t kTmemCols = BN < 32 ? 32 : BN;
  static constexpr uint32_t kIdesc = umma_idesc_bf16(128, BN);
};

template <int BN, int STAGES, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 2)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int K,
                   const typename Epi::Params p, uint32_t* __restrict__ err) {
  using Lay = GemmLayout<BN, STAGES>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the ring must start on a 1024-byte boundary (128-byte swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOffset);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_bar = empty + STAGES;
  uint64_t* drain_bar = acc_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* epi_smem = smem + Lay::kEpiOffset;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128;
  const int nk = K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Lay::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES && !mbar_wait_bounded(&empty[s], ((kb / STAGES) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        uint8_t* a_dst = smem + s * Lay::kStageBytes;
        uint8_t* b_dst = a_dst + Lay::kABytes;
        mbar_arrive_expect_tx(&full[s], Lay::kStageBytes);
        tma_load_2d(a_dst, &tmA, kb * kBK, m0, &full[s], pol_a);
        Epi::load_b(b_dst, &tmB, kb * kBK, p, &full[s], pol_b);
        issued = kb + 1;
      }
      // drain: the latest load of every stage must land before shared memory is released
      for (int kb = issued - STAGES > 0 ? issued - STAGES : 0; kb < issued; ++kb)
        mbar_wait_bounded(&full[kb % STAGES], (kb / STAGES) & 1, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait_bounded(&full[s], (kb / STAGES) & 1, err) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_addr(smem + s * Lay::kStageBytes);
        const uint32_t b_base = a_base + Lay::kABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          umma_bf16(tmem, umma_desc_sw128(a_base + k * 32), umma_desc_sw128(b_base + k * 32), Lay::kIdesc,
                    (kb | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(acc_bar);
    }
  } else {
    // epilogue warps 2..5
    const int q = warp & 3;                       // TMEM lane quarter of this warp
    const int row_local = q * 32 + lane;
    const bool ok = mbar_wait_bounded(acc_bar, 0, err) && !*abort_flag;
    tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 32, v);
        tmem_ld_wait();
        Epi::consume(p, epi_smem, m0, row_local, c, v);
      }
    }
    tc_fence_before();
  }
  // Epi::finish runs on all six warps (the producer and MMA warps are idle by now).
  __syncthreads();
  if (!*abort_flag) Epi::finish(p, epi_smem, m0, threadIdx.x);
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      // every MMA issued by this thread has completed once the drain barrier fires
      umma_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, err);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int BN, int STAGES, class Epi>
size_t tc_gemm_smem_bytes() {
  using Lay = GemmLayout<BN, STAGES>;
  return 1024 + Lay::kEpiOffset + Epi::kSmemBytes;
}

template <int BN, int STAGES, class Epi>
cudaError_t launch_tc_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int K, int grid_n,
                           const typename Epi::Params& p, uint32_t* err, cudaStream_t stream) {
  const size_t smem = tc_gemm_smem_bytes<BN, STAGES, Epi>();
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, Epi>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid((M + 127) / 128, grid_n);
  tc_gemm_kernel<BN, STAGES, Epi><<<grid, kGemmThreads, smem, stream>>>(tmA, tmB, K, p, err);
  return cudaGetLastError();
}

}  // namespace dflash2
