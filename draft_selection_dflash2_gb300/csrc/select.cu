// select.cu -- context gate and pairwise path-selector scores ("DFlash 2: Keep
// Drafting Parallel", "A Lightweight Path Selector", score equation
// S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>).
//
// gate             H = sigmoid(W_H h + b_H): one [B*L, d] x [d, 256] contraction on
//                  CTA pairs (tcgen05.mma.cta_group::2 + TMA, fp32 in TMEM), the
//                  K loop split into fp32 partials that a finishing kernel sums
//                  in a fixed order before the bias and the sigmoid.
// pair_kernel      one warp per block position at a time (positions strided
//                  over all warps of a one-CTA-per-SM grid): the warp copies
//                  the 16 predecessor rows of A, the 16 candidate rows of B
//                  (512 B each) and the position's gate partials into its own
//                  shared memory with 16-byte cp.async, forms H_t (and writes
//                  it), then takes the 16 x 16 x 256 products on the tensor
//                  cores (mma.sync m16n8k16, bf16 in, fp32 accumulate): B's rows
//                  are bf16 already, and G = A_pred (.) H_t in fp32 enters as
//                  the sum of two bf16 terms, its rounding and the rounding of
//                  the remainder, which carries G to about 2^-16 of its size.
#include "common.cuh"
#include "gemm_pair.cuh"
#include "launch.h"

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
  __device__ static int b_row(const Params&, int, int, int rank, int half) { return rank * half; }
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
constexpr int kPairWarps = 8;           // warps per CTA, one CTA per SM
constexpr int kRowPitch = kEmbed + 8;   // bf16 row pitch in shared memory (528 B: ldmatrix rows on distinct banks)

// one warp's shared memory: A rows, B rows (bf16), the gate partials and H (fp32)
__host__ __device__ inline size_t pair_warp_bytes(int ks) {
  return static_cast<size_t>(2 * kTopK * kRowPitch * 2) + static_cast<size_t>(ks) * kEmbed * 4 + kEmbed * 4;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

// D += A B, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two bf16 values (low, high halves of w) times (h0, h1) in fp32, split into
// the rounded products (hi) and the rounded remainders (lo).
__device__ __forceinline__ void scale_split(uint32_t w, float h0, float h1, uint32_t& hi, uint32_t& lo) {
  const float g0 = __uint_as_float(w << 16) * h0, g1 = __uint_as_float(w & 0xFFFF0000u) * h1;
  const __nv_bfloat162 hb = __floats2bfloat162_rn(g0, g1);
  const float r0 = g0 - __low2float(hb), r1 = g1 - __high2float(hb);
  const __nv_bfloat162 lb = __floats2bfloat162_rn(r0, r1);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
  lo = *reinterpret_cast<const uint32_t*>(&lb);
}

template <int KS>
__global__ void __launch_bounds__(kPairWarps * 32, 1) pair_kernel(const int32_t* __restrict__ cand_idx,
                                                                 const float* __restrict__ cand_val,
                                                                 const int32_t* __restrict__ last_verified,
                                                                 const float* __restrict__ gpart,
                                                                 const float* __restrict__ b_H,
                                                                 float* __restrict__ gate,
                                                                 const uint16_t* __restrict__ A,
                                                                 const uint16_t* __restrict__ Bt, int64_t L,
                                                                 int64_t V, int64_t npos, float* __restrict__ S,
                                                                 uint32_t* __restrict__ err) {
  extern __shared__ __align__(16) uint8_t pair_smem[];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = pair_smem + static_cast<size_t>(warp) * pair_warp_bytes(KS);
  uint16_t* As = reinterpret_cast<uint16_t*>(base);                  // [16][kRowPitch]
  uint16_t* Bs = As + kTopK * kRowPitch;                              // [16][kRowPitch]
  float* Ps = reinterpret_cast<float*>(Bs + kTopK * kRowPitch);       // [KS][256]
  float* Hs = Ps + KS * kEmbed;                                       // [256]
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kPairWarps;
  const int g = lane >> 2, c = lane & 3;
  for (int64_t pos = static_cast<int64_t>(blockIdx.x) * kPairWarps + warp; pos < npos; pos += nwarps) {
    const int64_t b = pos / L, t = pos - b * L;
    // lane q: predecessor id q (q < 16; the last verified token at t = 0) or candidate id q - 16
    int32_t id = lane < kTopK ? (t == 0 ? last_verified[b] : cand_idx[(pos - 1) * kTopK + lane])
                              : cand_idx[pos * kTopK + lane - kTopK];
    id = clamp_token(id, V, err);
    __syncwarp();   // the previous position's reads of this warp's buffers are done
    // row q: 32 16-byte pieces, lane = piece
#pragma unroll 4
    for (int q = 0; q < 2 * kTopK; ++q) {
      const int32_t rid = __shfl_sync(0xFFFFFFFFu, id, q);
      const uint16_t* src = (q < kTopK ? A : Bt) + static_cast<int64_t>(rid) * kEmbed + lane * 8;
      cp_async16((q < kTopK ? As + q * kRowPitch : Bs + (q - kTopK) * kRowPitch) + lane * 8, src);
    }
    // the position's gate partials ([KS][256], split-major)
#pragma unroll
    for (int k = 0; k < KS * 2; ++k) {
      const int item = lane + 32 * k;   // float4 item: split item / 64, piece item % 64
      cp_async16(Ps + item * 4, gpart + ((item >> 6) * npos + pos) * kEmbed + (item & 63) * 4);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    // H_t = sigmoid(sum of the KS partials in split order + b_H): lane owns channels 8 lane .. 8 lane + 7
    {
      float o[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4 z = *reinterpret_cast<const float4*>(Ps + lane * 8 + h * 4);
#pragma unroll
        for (int q = 1; q < KS; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(Ps + q * kEmbed + lane * 8 + h * 4);
          z.x += v.x;
          z.y += v.y;
          z.z += v.z;
          z.w += v.w;
        }
        const float zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = lane * 8 + h * 4 + j;
          o[h * 4 + j] = 1.0f / (1.0f + expf(-(zz[j] + (b_H ? b_H[ch] : 0.0f))));
        }
      }
      *reinterpret_cast<float4*>(Hs + lane * 8) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(Hs + lane * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
      *reinterpret_cast<float4*>(gate + pos * kEmbed + lane * 8) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(gate + pos * kEmbed + lane * 8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
    __syncwarp();
    // the products: S (16 x 16) = G (16 x 256) B^T, two 8-column tiles
    float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = ((lane >> 4) & 1) * 8;
    const int brow = (lane & 7) + ((lane >> 4) & 1) * 8, bcol = ((lane >> 3) & 1) * 8;
#pragma unroll 4
    for (int kk = 0; kk < kEmbed / 16; ++kk) {
      uint32_t af[4], bf[4];
      ldmatrix_x4(af, As + arow * kRowPitch + kk * 16 + acol);
      ldmatrix_x4(bf, Bs + brow * kRowPitch + kk * 16 + bcol);
      const float2 h01 = *reinterpret_cast<const float2*>(Hs + kk * 16 + 2 * c);
      const float2 h89 = *reinterpret_cast<const float2*>(Hs + kk * 16 + 2 * c + 8);
      uint32_t ahi[4], alo[4];
      scale_split(af[0], h01.x, h01.y, ahi[0], alo[0]);
      scale_split(af[1], h01.x, h01.y, ahi[1], alo[1]);
      scale_split(af[2], h89.x, h89.y, ahi[2], alo[2]);
      scale_split(af[3], h89.x, h89.y, ahi[3], alo[3]);
      mma_bf16(acc[0], ahi, bf[0], bf[1]);
      mma_bf16(acc[0], alo, bf[0], bf[1]);
      mma_bf16(acc[1], ahi, bf[2], bf[3]);
      mma_bf16(acc[1], alo, bf[2], bf[3]);
    }
    // S[i][j] = U_j + acc: rows g and g + 8, columns 8 nt + 2 c, + 1
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int j = nt * 8 + 2 * c;
      const float2 u = make_float2(cand_val[pos * kTopK + j], cand_val[pos * kTopK + j + 1]);   // 4-byte aligned only
      *reinterpret_cast<float2*>(S + (pos * kTopK + g) * kTopK + j) = make_float2(u.x + acc[nt][0], u.y + acc[nt][1]);
      *reinterpret_cast<float2*>(S + (pos * kTopK + g + 8) * kTopK + j) =
          make_float2(u.x + acc[nt][2], u.y + acc[nt][3]);
    }
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
  const int64_t ctas = (npos + kPairWarps - 1) / kPairWarps;
  const size_t smem = kPairWarps * pair_warp_bytes(8);
  cudaError_t se;
  switch (ks) {
    case 1: se = set_smem_limit<pair_kernel<1>>(smem); break;
    case 2: se = set_smem_limit<pair_kernel<2>>(smem); break;
    case 3: se = set_smem_limit<pair_kernel<3>>(smem); break;
    case 4: se = set_smem_limit<pair_kernel<4>>(smem); break;
    case 5: se = set_smem_limit<pair_kernel<5>>(smem); break;
    case 6: se = set_smem_limit<pair_kernel<6>>(smem); break;
    case 7: se = set_smem_limit<pair_kernel<7>>(smem); break;
    default: se = set_smem_limit<pair_kernel<8>>(smem); break;
  }
  if (se != cudaSuccess) return se;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas < num_sms ? ctas : num_sms), 1, 1);
  cfg.blockDim = dim3(kPairWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = kPairWarps * pair_warp_bytes(ks);
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
