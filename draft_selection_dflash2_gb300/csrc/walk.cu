// walk.cu -- the walk over precomputed pair scores ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector": starting from the last verified
// token, greedy follows the best successor at each step; sampling draws from
// the same scores).  This is the only sequential part of the draft-block head.
//
// One warp per sequence.  The warp first copies the sequence's whole score
// block S[b] ([L, 16, 16] fp32, 1 KB per position, one bulk asynchronous copy
// completing on an mbarrier) and its candidate ids ([L, 16] int32) into shared memory, and (sampled walk)
// computes the L Philox uniforms in parallel, one step per lane, so the L
// dependent steps touch neither global memory nor Philox.  Lane j (j < 16)
// owns successor slot j.
//   greedy : shuffle arg-max over (value, lowest slot), a NaN score below
//            every number (all NaN: slot 0).
//   sampled: everything in fp32 (the draw is an integer decided by floating
//            point): c = log2(e) / T, w_j = exp2_neg((S_j - max) * c), Z and the
//            CDF summed in slot order, u the Philox uniform of (b, t, stream 0)
//            (24 bits, exact in fp32), slot = smallest j with u Z < CDF_j,
//            q_j = w_j / Z.  exp2_neg follows Cody and Waite's reduction with a
//            degree-7 Taylor polynomial, and every step is a correctly rounded
//            IEEE operation (explicit _rn intrinsics, no contraction), so the
//            draw is reproducible by any implementation of the same steps.
//            A row with no positive weight (every score NaN or -inf) takes the
//            greedy slot, with q one-hot there.
#include "common.cuh"
#include "exp2.cuh"
#include "launch.h"
#include "philox.cuh"

namespace dflash2 {
namespace {

constexpr int kWalkWarps = 2;            // sequences per CTA (2 x 69 KB at L = 64)
constexpr int kMaxWalkL = 64;
// shared memory per sequence: S[b], its candidate ids and its L uniforms, rounded
// up to 4 floats so that every sequence's block (copied with 16-byte stores)
// starts on a 16-byte boundary
__host__ __device__ inline size_t walk_smem_floats(int64_t L) {
  return (static_cast<size_t>(L) * (kTopK * kTopK + kTopK + 1) + 3) & ~size_t(3);
}

__global__ void __launch_bounds__(kWalkWarps * 32)
    walk_kernel(const float* __restrict__ S, const int32_t* __restrict__ cand_idx, int64_t B,
                int64_t L, float temperature, uint64_t seed, uint64_t offset,
                int32_t* __restrict__ draft_tok, int32_t* __restrict__ draft_slot,
                float* __restrict__ draft_q, uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) float wsm[];
  __shared__ uint64_t bars[kWalkWarps];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kWalkWarps + warp;
  if (b >= B) return;
  float* sb = wsm + static_cast<size_t>(warp) * walk_smem_floats(L);
  int32_t* ids = reinterpret_cast<int32_t*>(sb + L * kTopK * kTopK);
  float* us = sb + L * (kTopK * kTopK + kTopK);
  // S[b] arrives by one bulk copy while the lanes load the ids and draw the uniforms
  uint64_t* bar = &bars[warp];
  if (lane == 0) {
    const uint32_t bytes = static_cast<uint32_t>(L * kTopK * kTopK * sizeof(float));
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sb, S + b * L * kTopK * kTopK, bytes, bar, l2_policy_evict_first());
  }
  {
    const int32_t* isrc = cand_idx + b * L * kTopK;   // 4-byte aligned only
    for (int i = lane; i < L * kTopK; i += 32) ids[i] = isrc[i];
    if (temperature > 0.0f)
      for (int t = lane; t < L; t += 32)
        us[t] = static_cast<float>(
            philox_uniform24(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 0, offset));
  }
  __syncwarp();
  if (!mbar_wait_bounded(bar, 0, err)) {
    mbar_wait_bounded(bar, 0, err);   // give the copy one more limit to land, then leave
    return;
  }

  const int j = lane & (kTopK - 1);
  const float cinv = temperature > 0.0f ? __fdiv_rn(1.44269504f, temperature) : 0.0f;
  int prev = 0;
  for (int64_t t = 0; t < L; ++t) {
    const float v = sb[(t * kTopK + prev) * kTopK + j];
    // arg-max under one total order, so every lane reaches the same slot: the
    // score's order image (NaN lowest, -0 == +0) above 15 - slot (lowest slot
    // first on ties); lanes 16..31 mirror 0..15
    uint64_t key = (static_cast<uint64_t>(score_order(v)) << 32) | static_cast<uint32_t>(kTopK - 1 - j);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) key = kmax(key, __shfl_xor_sync(0xFFFFFFFFu, key, o));
    const int bj = kTopK - 1 - static_cast<int>(key & 0xFu);
    const float bv = __shfl_sync(0xFFFFFFFFu, v, bj);
    int chosen;
    const int64_t q_at = (b * L + t) * kTopK + j;
    if (temperature <= 0.0f) {
      chosen = bj;
      if (draft_q && lane < kTopK) draft_q[q_at] = (j == chosen) ? 1.0f : 0.0f;
    } else {
      const float w = exp2_neg(__fmul_rn(__fsub_rn(v, bv), cinv));
      // Every lane gathers the 16 weights and repeats the (identical) slot-order
      // sums, so no broadcast is needed afterwards.
      float cdf[kTopK];
      float Z = 0.0f;
#pragma unroll
      for (int i = 0; i < kTopK; ++i) {
        Z = __fadd_rn(Z, __shfl_sync(0xFFFFFFFFu, w, i));
        cdf[i] = Z;
      }
      if (!(Z > 0.0f)) {
        // no positive weight (every score NaN or -inf): the greedy slot
        chosen = bj;
        if (draft_q && lane < kTopK) draft_q[q_at] = (j == chosen) ? 1.0f : 0.0f;
      } else {
        const float target = __fmul_rn(us[t], Z);
        int pick = -1;
#pragma unroll
        for (int i = kTopK - 1; i >= 0; --i)
          if (target < cdf[i]) pick = i;
        if (pick < 0) {
          // u Z below every partial sum cannot fail for u < 1; keep the last positive weight
          for (int i = kTopK - 1; i >= 0; --i)
            if (cdf[i] > (i > 0 ? cdf[i - 1] : 0.0f)) {
              pick = i;
              break;
            }
        }
        chosen = pick;
        if (draft_q && lane < kTopK) draft_q[q_at] = __fdiv_rn(w, Z);
      }
    }
    if (lane == 0) {
      draft_slot[b * L + t] = chosen;
      draft_tok[b * L + t] = ids[t * kTopK + chosen];
    }
    prev = chosen;
  }
}

}  // namespace

cudaError_t launch_walk(const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                        float temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                        int32_t* draft_slot, float* draft_q, uint32_t* err, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kWalkWarps) * walk_smem_floats(L) * sizeof(float);
  {
    const cudaError_t e = set_smem_limit<walk_kernel>(kWalkWarps * walk_smem_floats(kMaxWalkL) * sizeof(float));
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>((B + kWalkWarps - 1) / kWalkWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kWalkWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, walk_kernel, S, cand_idx, B, L, temperature, seed, offset, draft_tok, draft_slot,
                            draft_q, err);
}

}  // namespace dflash2
