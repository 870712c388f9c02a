// viterbi.cu -- the exact best path over the pair scores: the max-sum
// recurrence on the chain of 16 x 16 score matrices of "A Lightweight Path
// Selector" ("DFlash 2: Keep Drafting Parallel"), the exact counterpart of its
// greedy walk.  Scores add in fp32 from left to right; ties go to the lowest
// predecessor slot and, at the end, to the lowest final slot.
//
// One warp per sequence.  The warp copies S[b] ([L, 16, 16] fp32, one bulk
// asynchronous copy completing on an mbarrier) and its candidate ids into
// shared memory.  Lane j (j < 16) holds V[j],
// the best score of a path ending in slot j; at each step it forms
// V[i] + S[t][i][j] for i = 0..15 in order, keeps the first strict maximum, and
// records that predecessor as a byte in shared memory.  Lane 0 then takes the
// lowest slot of the best final score and follows the recorded predecessors
// back to t = 0.
#include "common.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

constexpr int kViterbiWarps = 2;         // sequences per CTA (2 x 70 KB at L = 64)
constexpr int kViterbiMaxL = 64;
// shared memory per sequence: S[b], its candidate ids and L x 16 predecessor
// bytes, rounded up to 4 floats so that every sequence's block (written with
// 16-byte stores) starts on a 16-byte boundary
__host__ __device__ inline size_t viterbi_smem_floats(int64_t L) {
  return (static_cast<size_t>(L) * (kTopK * kTopK + kTopK + kTopK / 4) + 3) & ~size_t(3);
}

__global__ void __launch_bounds__(kViterbiWarps * 32)
    walk_viterbi_kernel(const float* __restrict__ S, const int32_t* __restrict__ cand_idx, int64_t B, int64_t L,
                        int32_t* __restrict__ draft_tok, int32_t* __restrict__ draft_slot,
                        float* __restrict__ score, uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) float wsm[];
  __shared__ uint64_t bars[kViterbiWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kViterbiWarps + warp;
  if (b >= B) return;
  float* sb = wsm + static_cast<size_t>(warp) * viterbi_smem_floats(L);
  int32_t* ids = reinterpret_cast<int32_t*>(sb + L * kTopK * kTopK);
  uint8_t* back = reinterpret_cast<uint8_t*>(sb + L * (kTopK * kTopK + kTopK));
  // S[b] arrives by one bulk copy while the lanes load the ids
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
  }
  __syncwarp();
  if (!mbar_wait_bounded(bar, 0, err)) {
    mbar_wait_bounded(bar, 0, err);   // give the copy one more limit to land, then leave
    return;
  }
  const int j = lane & (kTopK - 1);
  float V = sb[j];   // t = 0: row 0 (the last verified token)
  for (int64_t t = 1; t < L; ++t) {
    const float* st = sb + t * kTopK * kTopK;
    float best = __fadd_rn(__shfl_sync(0xFFFFFFFFu, V, 0), st[j]);
    int arg = 0;
#pragma unroll
    for (int i = 1; i < kTopK; ++i) {
      const float v = __fadd_rn(__shfl_sync(0xFFFFFFFFu, V, i), st[i * kTopK + j]);
      if (v > best) {
        best = v;
        arg = i;
      }
    }
    if (lane < kTopK) back[t * kTopK + j] = static_cast<uint8_t>(arg);
    V = best;
  }
  __syncwarp();
  float fin[kTopK];
#pragma unroll
  for (int i = 0; i < kTopK; ++i) fin[i] = __shfl_sync(0xFFFFFFFFu, V, i);
  if (lane == 0) {
    int jj = 0;
    float fb = fin[0];
#pragma unroll
    for (int i = 1; i < kTopK; ++i)
      if (fin[i] > fb) {
        fb = fin[i];
        jj = i;
      }
    if (score) score[b] = fb;
    for (int64_t t = L - 1; t >= 0; --t) {
      draft_slot[b * L + t] = jj;
      draft_tok[b * L + t] = ids[t * kTopK + jj];
      if (t > 0) jj = back[t * kTopK + jj];
    }
  }
}

}  // namespace

cudaError_t launch_walk_viterbi(const float* S, const int32_t* cand_idx, int64_t B, int64_t L, int32_t* draft_tok,
                                int32_t* draft_slot, float* score, uint32_t* err, cudaStream_t stream) {
  if (L > kViterbiMaxL) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kViterbiWarps) * viterbi_smem_floats(L) * sizeof(float);
  {
    const cudaError_t e =
        set_smem_limit<walk_viterbi_kernel>(kViterbiWarps * viterbi_smem_floats(kViterbiMaxL) * sizeof(float));
    if (e != cudaSuccess) return e;
  }
  const unsigned grid = static_cast<unsigned>((B + kViterbiWarps - 1) / kViterbiWarps);
  walk_viterbi_kernel<<<grid, kViterbiWarps * 32, smem, stream>>>(S, cand_idx, B, L, draft_tok, draft_slot, score,
                                                                      err);
  return cudaGetLastError();
}

}  // namespace dflash2
