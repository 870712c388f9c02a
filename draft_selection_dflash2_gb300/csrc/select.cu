// select.cu -- context gate and pairwise path-selector scores ("DFlash 2: Keep
// Drafting Parallel", "A Lightweight Path Selector", score equation
// S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>).
//
// gate             H = sigmoid(W_H h + b_H): one [B*L, d] x [d, 256] contraction on
//                  the tensor cores (tcgen05 + TMA, fp32 in TMEM, K split over a
//                  cluster and reduced in distributed shared memory), sigmoid
//                  fused in the epilogue.
// pair_kernel      persistent, block positions strided over the CTAs: for each
//                  (b, t) gathers the 16 predecessor rows of A and the 16
//                  candidate rows of B (512 B each) with 16-byte loads, forms
//                  G = A_pred (.) H_t in fp32 shared memory and computes the
//                  16 x 16 x 256 products (pair_math.cuh); the next position's
//                  rows are gathered while the products run.
#include "common.cuh"
#include "gemm_splitk.cuh"
#include "launch.h"
#include "pair_math.cuh"

namespace dflash2 {
namespace {

// ---------------------------------------------------------------------------
// gate: H = sigmoid(h W_H^T + b) on the tensor cores (gemm_splitk.cuh): 128
// positions x 128 of the 256 gate channels per tile, K split over a cluster of
// up to 4 CTAs (small clusters place readily next to other kernels' CTAs),
// partial sums reduced through distributed shared memory, sigmoid in the
// epilogue.
// ---------------------------------------------------------------------------
constexpr int kGateBN = 128;

struct GateEpi {
  struct Params {
    float* gate;          // [M, 256]
    const float* bias;    // [256] or null
    int M;
  };
  __host__ __device__ static int sub_n(int BN) { return BN; }

  __device__ static void load_b(void* dst, const CUtensorMap* tm, int k, int n_tile, const Params&, uint64_t* bar,
                                uint64_t pol) {
    tma_load_2d(dst, tm, k, n_tile * kGateBN, bar, pol);
  }
  __device__ static __forceinline__ void finish(const Params& p, const SplitKShape& sh, uint8_t* region, uint64_t*,
                                                int m0, int n_tile, int rank, int tid, uint32_t*) {
    const SkPartials parts(reinterpret_cast<const float*>(region), sh.ks, sk_partial_pitch(sh.BN));
    const int rows_per = 128 / sh.ks;
    const int r0 = rank * rows_per;
    const int c0 = n_tile * kGateBN;
    const int total = rows_per * (kGateBN / 4);
    for (int e = tid; e < total; e += kSkThreads) {
      const int lr = e / (kGateBN / 4), c4 = (e % (kGateBN / 4)) * 4;
      const int m = m0 + r0 + lr;
      if (m >= p.M) continue;
      const float4 z = parts.sum4(lr, c4);
      const float zz[4] = {z.x, z.y, z.z, z.w};
      float o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = 1.0f / (1.0f + expf(-(zz[j] + (p.bias ? p.bias[c0 + c4 + j] : 0.0f))));
      *reinterpret_cast<float4*>(p.gate + static_cast<int64_t>(m) * kEmbed + c0 + c4) =
          make_float4(o[0], o[1], o[2], o[3]);
    }
  }
};

// ---------------------------------------------------------------------------
// pair scores
// ---------------------------------------------------------------------------
constexpr int kPairCtasPerSm = 3;

// One position's gathered operands, in registers: thread tid's items are rows
// tid / 32 + 8 it (it = 0, 1: A rows; 2, 3: B rows), 16-byte chunk tid % 32,
// plus the H_t chunk the A items are scaled by.
struct PairStage {
  uint4 raw[4];
  float4 h0, h1;
};

__device__ __forceinline__ void pair_issue(PairStage& st, const int32_t* ids, const uint16_t* __restrict__ A,
                                           const uint16_t* __restrict__ Bt, const float* __restrict__ gate,
                                           int64_t pos, int tid) {
  const int ch = tid & 31;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int row = (tid >> 5) + 8 * it;   // 0..15: A (predecessors), 16..31: B (candidates)
    const uint16_t* src = row < kTopK ? A + static_cast<int64_t>(ids[row]) * kEmbed
                                      : Bt + static_cast<int64_t>(ids[row]) * kEmbed;
    st.raw[it] = *reinterpret_cast<const uint4*>(src + ch * 8);
  }
  const float* Ht = gate + pos * kEmbed + ch * 8;
  st.h0 = *reinterpret_cast<const float4*>(Ht);
  st.h1 = *reinterpret_cast<const float4*>(Ht + 4);
}

// G = A_pred (.) H_t and Bc = B_cand in fp32 shared memory.
__device__ __forceinline__ void pair_store(const PairStage& st, float (*G)[kEmbed], float (*Bc)[kEmbed], int tid) {
  const int ch = tid & 31;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int row = (tid >> 5) + 8 * it;
    const uint32_t w[4] = {st.raw[it].x, st.raw[it].y, st.raw[it].z, st.raw[it].w};
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = bf16_bits_to_float(w[q] & 0xFFFFu);
      f[2 * q + 1] = bf16_bits_to_float(w[q] >> 16);
    }
    if (row < kTopK) {
      f[0] *= st.h0.x; f[1] *= st.h0.y; f[2] *= st.h0.z; f[3] *= st.h0.w;
      f[4] *= st.h1.x; f[5] *= st.h1.y; f[6] *= st.h1.z; f[7] *= st.h1.w;
      *reinterpret_cast<float4*>(&G[row][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&G[row][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      *reinterpret_cast<float4*>(&Bc[row - kTopK][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&Bc[row - kTopK][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
}

// Persistent: CTA c takes positions c, c + grid, ...  While the products of
// one position run, the rows of the next are in flight in registers and the
// ids of the one after that are loading.
__global__ void __launch_bounds__(256, kPairCtasPerSm) pair_kernel(const int32_t* __restrict__ cand_idx,
                                                                   const float* __restrict__ cand_val,
                                                                   const int32_t* __restrict__ last_verified,
                                                                   const float* __restrict__ gate,
                                                                   const uint16_t* __restrict__ A,
                                                                   const uint16_t* __restrict__ Bt, int64_t L,
                                                                   int64_t V, int64_t npos, float* __restrict__ S,
                                                                   uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ __align__(16) float G[kTopK][kEmbed];    // A[pred_i] (.) H_t
  __shared__ __align__(16) float Bc[kTopK][kEmbed];   // B[cand_j]
  __shared__ int32_t ids[2][2 * kTopK];               // pred (0..15) and cand (16..31) ids of coming positions
  const int tid = threadIdx.x;
  const int64_t stride = gridDim.x;
  int64_t pos = blockIdx.x;
  if (pos >= npos) return;
  // thread q < 32: predecessor (q < 16) or candidate (q >= 16) id q of position p
  auto load_id = [&](int64_t p) -> int32_t {
    const int64_t b = p / L, t = p % L;
    const int32_t v = tid < kTopK ? (t == 0 ? last_verified[b] : cand_idx[(p - 1) * kTopK + tid])
                                  : cand_idx[p * kTopK + tid - kTopK];
    return clamp_token(v, V, err);
  };
  if (tid < 2 * kTopK) ids[0][tid] = load_id(pos);
  int32_t next_id = tid < 2 * kTopK && pos + stride < npos ? load_id(pos + stride) : 0;
  __syncthreads();
  PairStage st;
  pair_issue(st, ids[0], A, Bt, gate, pos, tid);
  int buf = 0;
  for (; pos < npos; pos += stride) {
    const int64_t pn = pos + stride;
    pair_store(st, G, Bc, tid);
    if (tid < 2 * kTopK) ids[buf ^ 1][tid] = next_id;
    next_id = tid < 2 * kTopK && pn + stride < npos ? load_id(pn + stride) : 0;
    __syncthreads();   // G, Bc and the next position's ids are in place
    if (pn < npos) pair_issue(st, ids[buf ^ 1], A, Bt, gate, pn, tid);
    pair_products(G, Bc, cand_val, S, pos, tid);
    __syncthreads();   // G and Bc are free again
    buf ^= 1;
  }
}

}  // namespace

cudaError_t launch_gate(const uint16_t* hs, const uint16_t* W_H, const float* b_H, int64_t M,
                        int64_t d, float* gate, uint32_t* err, int num_sms, cudaStream_t stream) {
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  SplitKShape sh;
  sh.M = static_cast<int>(M);
  sh.K = static_cast<int>(d);
  sh.BN = kGateBN;
  sh.n_tiles = kEmbed / kGateBN;
  sh.m_tiles = static_cast<int>((M + 127) / 128);
  sh.ks = sk_choose_ks(sh.n_tiles * sh.m_tiles, sh.K / kBK, num_sms);
  if (sh.ks > 4) sh.ks = 4;
  sh.tmem_cols = kGateBN;
  if (!sk_plan(sh)) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, hs, M, d, d, 128) || !make_tmap_bf16_2d(&tb, W_H, kEmbed, d, d, kGateBN))
    return cudaErrorInvalidValue;
  GateEpi::Params p{gate, b_H, static_cast<int>(M)};
  return launch_splitk_gemm<GateEpi>(ta, tb, sh, p, err, stream);
}

cudaError_t launch_pair_scores(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* last_verified, const float* gate, const uint16_t* A,
                               const uint16_t* Bt, int64_t B, int64_t L, int64_t V, float* S,
                               uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t npos = B * L;
  const int64_t slots = static_cast<int64_t>(kPairCtasPerSm) * num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(npos < slots ? npos : slots), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pair_kernel, cand_idx, cand_val, last_verified, gate, A, Bt, L, V, npos, S, err);
}

}  // namespace dflash2
