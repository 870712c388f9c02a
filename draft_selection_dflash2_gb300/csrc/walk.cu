// walk.cu -- the walk over precomputed pair scores ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector": starting from the last verified
// token, greedy follows the best successor at each step; sampling draws from
// the same scores).  This is the only sequential part of the draft-block head.
//
// One CTA per sequence, in two phases.  The successor chosen from predecessor
// slot p at position t depends only on row S[b, t, p, :] and on position t's
// uniform, never on the path, so every (t, p) row is resolved at once (one
// thread per row) and the L dependent steps become L lookups in shared memory.
//   greedy : arg-max over (value, lowest slot), a NaN score below every
//            number (all NaN: slot 0).
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
// Then thread 0 follows the chosen slots from slot 0 (the last verified
// token) and every thread writes its share of the outputs: slots, tokens and
// q, recomputed for the path's rows from the row's stored maximum and Z with
// the same operations.
#include "common.cuh"
#include "exp2.cuh"
#include "launch.h"
#include "philox.cuh"

namespace dflash2 {
namespace {

constexpr int kWalkThreads = 256;
constexpr int kMaxWalkL = 64;
// shared memory: S[b] ([L, 16, 16] fp32) and, per row, its maximum, Z and the
// chosen slot; then the path
__host__ __device__ inline size_t walk_smem_bytes(int64_t L) {
  return static_cast<size_t>(L) * kTopK * (kTopK * 4 + 4 + 4 + 4) + static_cast<size_t>(L) * 4;
}

__global__ void __launch_bounds__(kWalkThreads)
    walk_kernel(const float* __restrict__ S, const int32_t* __restrict__ cand_idx, int64_t B,
                int64_t L, float temperature, uint64_t seed, uint64_t offset,
                int32_t* __restrict__ draft_tok, int32_t* __restrict__ draft_slot,
                float* __restrict__ draft_q) {
  extern __shared__ __align__(16) float wsm[];
  pdl_wait();
  pdl_launch_dependents();
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x;
  const int rows = static_cast<int>(L) * kTopK;
  float* Ss = wsm;                          // [rows][16]
  float* row_max = Ss + rows * kTopK;       // [rows]
  float* row_z = row_max + rows;            // [rows]
  int32_t* chosen = reinterpret_cast<int32_t*>(row_z + rows);   // [rows]
  int32_t* path = chosen + rows;            // [L]
  const bool sampled = temperature > 0.0f;
  const float cinv = sampled ? __fdiv_rn(1.44269504f, temperature) : 0.0f;
  const float4* src = reinterpret_cast<const float4*>(S + b * L * kTopK * kTopK);
  for (int r = tid; r < rows; r += kWalkThreads) {
    float v[kTopK];
#pragma unroll
    for (int k = 0; k < kTopK / 4; ++k) {
      const float4 q = __ldg(src + r * (kTopK / 4) + k);
      v[4 * k] = q.x;
      v[4 * k + 1] = q.y;
      v[4 * k + 2] = q.z;
      v[4 * k + 3] = q.w;
      reinterpret_cast<float4*>(Ss + r * kTopK)[k] = q;
    }
    // arg-max under one total order: the score's order image (NaN lowest,
    // -0 == +0) above 15 - slot (lowest slot first on ties)
    uint64_t key = 0ull;
#pragma unroll
    for (int j = 0; j < kTopK; ++j)
      key = kmax(key, (static_cast<uint64_t>(score_order(v[j])) << 32) | static_cast<uint32_t>(kTopK - 1 - j));
    const int bj = kTopK - 1 - static_cast<int>(key & 0xFu);
    float bv = v[0];
#pragma unroll
    for (int j = 1; j < kTopK; ++j)
      if (j == bj) bv = v[j];
    int pick = bj;
    float Z = 0.0f;
    if (sampled) {
      float cdf[kTopK];
#pragma unroll
      for (int j = 0; j < kTopK; ++j) {
        Z = __fadd_rn(Z, exp2_neg(__fmul_rn(__fsub_rn(v[j], bv), cinv)));
        cdf[j] = Z;
      }
      if (Z > 0.0f) {
        const int t = r / kTopK;
        const float u = static_cast<float>(
            philox_uniform24(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 0, offset));
        const float target = __fmul_rn(u, Z);
        pick = -1;
#pragma unroll
        for (int i = kTopK - 1; i >= 0; --i)
          if (target < cdf[i]) pick = i;
        if (pick < 0) {
          // u Z below every partial sum cannot fail for u < 1; keep the last positive weight
          float below = 0.0f;
#pragma unroll
          for (int i = 0; i < kTopK; ++i) {
            if (cdf[i] > below) pick = i;
            below = cdf[i];
          }
        }
      }
    }
    row_max[r] = bv;
    row_z[r] = Z;
    chosen[r] = pick;
  }
  __syncthreads();
  if (tid == 0) {
    int prev = 0;
    for (int t = 0; t < L; ++t) {
      prev = chosen[t * kTopK + prev];
      path[t] = prev;
    }
  }
  __syncthreads();
  for (int e = tid; e < rows; e += kWalkThreads) {
    const int t = e / kTopK, j = e % kTopK;
    const int slot = path[t];
    const int r = t * kTopK + (t > 0 ? path[t - 1] : 0);   // the row the step read
    if (j == 0) {
      draft_slot[b * L + t] = slot;
      draft_tok[b * L + t] = cand_idx[(b * L + t) * kTopK + slot];
    }
    if (draft_q) {
      float q;
      const float Z = row_z[r];
      if (sampled && Z > 0.0f)
        q = __fdiv_rn(exp2_neg(__fmul_rn(__fsub_rn(Ss[r * kTopK + j], row_max[r]), cinv)), Z);
      else
        q = j == slot ? 1.0f : 0.0f;
      draft_q[(b * L + t) * kTopK + j] = q;
    }
  }
}

}  // namespace

cudaError_t launch_walk(const float* S, const int32_t* cand_idx, int64_t B, int64_t L,
                        float temperature, uint64_t seed, uint64_t offset, int32_t* draft_tok,
                        int32_t* draft_slot, float* draft_q, uint32_t* err, cudaStream_t stream) {
  (void)err;   // nothing in the walk waits or can fail on the device
  if (L > kMaxWalkL) return cudaErrorInvalidValue;
  if (B == 0 || L == 0) return cudaSuccess;
  {
    const cudaError_t e = set_smem_limit<walk_kernel>(walk_smem_bytes(kMaxWalkL));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(kWalkThreads, 1, 1);
  cfg.dynamicSmemBytes = walk_smem_bytes(L);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, walk_kernel, S, cand_idx, B, L, temperature, seed, offset, draft_tok, draft_slot,
                            draft_q);
}

}  // namespace dflash2
