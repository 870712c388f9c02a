// select.cu -- context gate and pairwise path-selector scores ("DFlash 2: Keep
// Drafting Parallel", "A Lightweight Path Selector", score equation
// S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>).
//
// gate             H = sigmoid(W_H h + b_H): one [B*L, d] x [d, 256] contraction on
//                  CTA pairs (tcgen05.mma.cta_group::2 + TMA, fp32 in TMEM), the
//                  K loop split into fp32 partials that a finishing kernel sums
//                  in a fixed order before the bias and the sigmoid.
// pair_kernel      persistent, block positions strided over the CTAs: for each
//                  (b, t) gathers the 16 predecessor rows of A and the 16
//                  candidate rows of B (512 B each) with 16-byte loads and the
//                  position's gate partials, forms H_t (and writes it), G =
//                  A_pred (.) H_t in fp32 shared memory and computes the
//                  16 x 16 x 256 products (pair_math.cuh); the next position's
//                  rows and partials are gathered while the products run.
#include "common.cuh"
#include "gemm_pair.cuh"
#include "launch.h"
#include "pair_math.cuh"

namespace dflash2 {
namespace {

// ---------------------------------------------------------------------------
// gate: the contraction h W_H^T on CTA pairs (gemm_pair.cuh): 256 positions x
// the 256 gate channels per pair tile, the K loop split ks ways into fp32
// partials.  The pair kernel sums a position's partials in split order (the
// same bits on every run), adds the bias, applies the sigmoid and writes H.
// ---------------------------------------------------------------------------
struct GateShape {
  static constexpr int kSubs = 1;
  struct Params {
    int unused;
  };
  __device__ static int b_row(const Params&, int, int) { return 0; }
  __device__ static bool valid(const Params&, int, int) { return true; }
  __device__ static int out_col(const Params&, int, int c) { return c; }
};

PairGemmShape gate_plan(int64_t M, int64_t d, int num_sms) {
  PairGemmShape sh;
  sh.M = static_cast<int>(M);
  sh.K = static_cast<int>(d);
  sh.N = kEmbed;
  sh.BN = kEmbed;
  sh.n_tiles = 1;
  sh.m_pairs = static_cast<int>((M + 255) / 256);
  sh.ks = pg_choose_ks(sh.m_pairs, sh.K / kBK, num_sms);
  sh.tmem_cols = kEmbed;
  return sh;
}

// ---------------------------------------------------------------------------
// pair scores
// ---------------------------------------------------------------------------
constexpr int kPairCtasPerSm = 3;

// One position's gathered operands, in registers: thread tid's items are rows
// tid / 32 + 8 it (it = 0, 1: A rows; 2, 3: B rows), 16-byte chunk tid % 32,
// plus float4 items tid and tid + 256 of the position's gate partials
// ([KS][256], split-major).
template <int KS>
struct PairStage {
  static constexpr int kItems = (KS * kEmbed / 4 + 255) / 256;
  uint4 raw[4];
  float4 part[kItems];
};

template <int KS>
__device__ __forceinline__ void pair_issue(PairStage<KS>& st, const int32_t* ids, const uint16_t* __restrict__ A,
                                           const uint16_t* __restrict__ Bt, const float* __restrict__ gpart,
                                           int64_t M, int64_t pos, int tid) {
  const int ch = tid & 31;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int row = (tid >> 5) + 8 * it;   // 0..15: A (predecessors), 16..31: B (candidates)
    const uint16_t* src = row < kTopK ? A + static_cast<int64_t>(ids[row]) * kEmbed
                                      : Bt + static_cast<int64_t>(ids[row]) * kEmbed;
    st.raw[it] = *reinterpret_cast<const uint4*>(src + ch * 8);
  }
#pragma unroll
  for (int k = 0; k < PairStage<KS>::kItems; ++k) {
    const int item = tid + 256 * k;   // split item / 64, float4 item % 64
    if (item < KS * kEmbed / 4)
      st.part[k] = __ldcg(reinterpret_cast<const float4*>(gpart + ((item >> 6) * M + pos) * kEmbed) + (item & 63));
  }
}

// H_t = sigmoid(sum of the KS partials in split order + b_H) into Hs (shared)
// and the gate output; whole-CTA call, two barriers.
template <int KS>
__device__ __forceinline__ void pair_gate(const PairStage<KS>& st, float* Pb, float* Hs, const float* __restrict__ b_H,
                                          float* __restrict__ gate, int64_t pos, int tid) {
#pragma unroll
  for (int k = 0; k < PairStage<KS>::kItems; ++k) {
    const int item = tid + 256 * k;
    if (item < KS * kEmbed / 4) *reinterpret_cast<float4*>(Pb + item * 4) = st.part[k];
  }
  __syncthreads();
  if (tid < kEmbed / 4) {
    float4 z = *reinterpret_cast<const float4*>(Pb + tid * 4);
#pragma unroll
    for (int q = 1; q < KS; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(Pb + q * kEmbed + tid * 4);
      z.x += v.x;
      z.y += v.y;
      z.z += v.z;
      z.w += v.w;
    }
    const float zz[4] = {z.x, z.y, z.z, z.w};
    float o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = 1.0f / (1.0f + expf(-(zz[j] + (b_H ? b_H[tid * 4 + j] : 0.0f))));
    const float4 h = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(Hs + tid * 4) = h;
    *reinterpret_cast<float4*>(gate + pos * kEmbed + tid * 4) = h;
  }
  __syncthreads();
}

// G = A_pred (.) H_t and Bc = B_cand in fp32 shared memory.
template <int KS>
__device__ __forceinline__ void pair_store(const PairStage<KS>& st, const float* Hs, float (*G)[kEmbed],
                                           float (*Bc)[kEmbed], int tid) {
  const int ch = tid & 31;
  const float4 h0 = *reinterpret_cast<const float4*>(Hs + ch * 8), h1 = *reinterpret_cast<const float4*>(Hs + ch * 8 + 4);
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
      f[0] *= h0.x; f[1] *= h0.y; f[2] *= h0.z; f[3] *= h0.w;
      f[4] *= h1.x; f[5] *= h1.y; f[6] *= h1.z; f[7] *= h1.w;
      *reinterpret_cast<float4*>(&G[row][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&G[row][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      *reinterpret_cast<float4*>(&Bc[row - kTopK][ch * 8]) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(&Bc[row - kTopK][ch * 8 + 4]) = make_float4(f[4], f[5], f[6], f[7]);
    }
  }
}

// Persistent: CTA c takes positions c, c + grid, ...  While the products of
// one position run, the rows and gate partials of the next are in flight in
// registers and the ids of the one after that are loading.
template <int KS>
__global__ void __launch_bounds__(256, kPairCtasPerSm) pair_kernel(const int32_t* __restrict__ cand_idx,
                                                                   const float* __restrict__ cand_val,
                                                                   const int32_t* __restrict__ last_verified,
                                                                   const float* __restrict__ gpart,
                                                                   const float* __restrict__ b_H,
                                                                   float* __restrict__ gate,
                                                                   const uint16_t* __restrict__ A,
                                                                   const uint16_t* __restrict__ Bt, int64_t L,
                                                                   int64_t V, int64_t npos, float* __restrict__ S,
                                                                   uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ __align__(16) float G[kTopK][kEmbed];    // A[pred_i] (.) H_t
  __shared__ __align__(16) float Bc[kTopK][kEmbed];   // B[cand_j]
  __shared__ __align__(16) float Pb[KS * kEmbed];     // the position's gate partials
  __shared__ __align__(16) float Hs[kEmbed];          // H_t
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
  PairStage<KS> st;
  pair_issue<KS>(st, ids[0], A, Bt, gpart, npos, pos, tid);
  int buf = 0;
  for (; pos < npos; pos += stride) {
    const int64_t pn = pos + stride;
    pair_gate<KS>(st, Pb, Hs, b_H, gate, pos, tid);
    pair_store<KS>(st, Hs, G, Bc, tid);
    if (tid < 2 * kTopK) ids[buf ^ 1][tid] = next_id;
    next_id = tid < 2 * kTopK && pn + stride < npos ? load_id(pn + stride) : 0;
    __syncthreads();   // G, Bc and the next position's ids are in place
    if (pn < npos) pair_issue<KS>(st, ids[buf ^ 1], A, Bt, gpart, npos, pn, tid);
    pair_products(G, Bc, cand_val, S, pos, tid);
    __syncthreads();   // G and Bc are free again
    buf ^= 1;
  }
}

}  // namespace

size_t gate_workspace_bytes(int64_t B, int64_t L, int64_t d, int num_sms) {
  const PairGemmShape sh = gate_plan(B * L, d, num_sms);
  return static_cast<size_t>(sh.ks) * static_cast<size_t>(B * L) * kEmbed * sizeof(float);
}

cudaError_t launch_gate(const uint16_t* hs, const uint16_t* W_H, const float* b_H, int64_t M,
                        int64_t d, float* gate, void* workspace, uint32_t* err, int num_sms, cudaStream_t stream) {
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  PairGemmShape sh = gate_plan(M, d, num_sms);
  if (!pg_plan(sh)) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, hs, M, d, d, 128) || !make_tmap_bf16_2d(&tb, W_H, kEmbed, d, d, kEmbed / 2))
    return cudaErrorInvalidValue;
  return launch_pair_gemm<GateShape>(ta, tb, sh, GateShape::Params{0}, static_cast<float*>(workspace), err, stream);
}

cudaError_t launch_pair_scores(const int32_t* cand_idx, const float* cand_val,
                               const int32_t* last_verified, const float* gate_part, const float* b_H, float* gate,
                               int64_t d, const uint16_t* A, const uint16_t* Bt, int64_t B, int64_t L, int64_t V,
                               float* S, uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t npos = B * L;
  const int ks = gate_plan(npos, d, num_sms).ks;
  const int64_t slots = static_cast<int64_t>(kPairCtasPerSm) * num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(npos < slots ? npos : slots), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define DFLASH2_PAIR_LAUNCH(KS_) \
  cudaLaunchKernelEx(&cfg, pair_kernel<KS_>, cand_idx, cand_val, last_verified, gate_part, b_H, gate, A, Bt, L, V, \
                     npos, S, err)
  switch (ks) {
    case 1: return DFLASH2_PAIR_LAUNCH(1);
    case 2: return DFLASH2_PAIR_LAUNCH(2);
    case 3: return DFLASH2_PAIR_LAUNCH(3);
    case 4: return DFLASH2_PAIR_LAUNCH(4);
    case 5: return DFLASH2_PAIR_LAUNCH(5);
    case 6: return DFLASH2_PAIR_LAUNCH(6);
    case 7: return DFLASH2_PAIR_LAUNCH(7);
    default: return DFLASH2_PAIR_LAUNCH(8);
  }
#undef DFLASH2_PAIR_LAUNCH
}

}  // namespace dflash2
