// verify.cu -- block verification against the target's logits ("DFlash 2: Keep
// Drafting Parallel": the target checks the whole block in one forward pass;
// "A Lightweight Path Selector": rejection sampling restores the exact target
// distribution; Table 1's note: the acceptance length includes the verifier's
// next token).
//
// Three launches:
//   init      first_reject[b] := L (stored in accept_len, which the caller owns)
//   rows      one CTA per target row (b, t), scheduled t-major.  A CTA first reads
//             first_reject[b]; when an earlier position already rejected, the
//             row cannot matter and the CTA returns without reading it, so most
//             rows past the accepted prefix are never streamed.
//               T = 0: arg-max (lowest id on ties) -> out_tok[b, t]; a mismatch
//                      lowers first_reject[b] with atomicMin.
//               T > 0: online softmax statistics (max, Z) of the row with
//                      fp32 ex2 and fp64 combination; the accept test
//                      u1 q Z < exp((l_x - max)/T); a rejection draws from the
//                      residual max(0, e_v - q_v Z) by a blocked inverse CDF in id
//                      order (fp64 prefix sums); row L draws the bonus token.
//   finalize  n = first_reject[b]; out_tok = draft[0..n-1], row n's token, -1...;
//             accept_len[b] = n + 1.
#include "common.cuh"
#include "launch.h"
#include "philox.cuh"

namespace dflash2 {
namespace {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t lane_bits(const uint4& v, int k) {
  const uint32_t w = (k < 4) ? ((k < 2) ? v.x : v.y) : ((k < 6) ? v.z : v.w);
  return (k & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ uint32_t vec_max_bits(uint4 v) {
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&v.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v.y);
  __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&v.z);
  __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&v.w);
  const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
  const __nv_bfloat16 mm = __hmax(__low2bfloat16(m), __high2bfloat16(m));
  return static_cast<uint32_t>(__bfloat16_as_ushort(mm));
}

// ---------------------------------------------------------------------------
// block reductions
// ---------------------------------------------------------------------------
struct VerifySmem {
  uint64_t key[kVWarps];
  float m[kVWarps];
  double z[kVWarps];
  double scan[kVThreads];
  int32_t cand[kTopK];
  double candr[kTopK];        // residual weight of each candidate (unnormalized)
  float row_max;
  double row_z;
  int skip;
  int token;
};

__device__ uint64_t block_max_key(VerifySmem& s, uint64_t k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = kmax(k, __shfl_xor_sync(0xFFFFFFFFu, k, o));
  if (lane == 0) s.key[warp] = k;
  __syncthreads();
  uint64_t r = s.key[0];
#pragma unroll
  for (int w = 1; w < kVWarps; ++w) r = kmax(r, s.key[w]);
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
__global__ void verify_init_kernel(int32_t* first_reject, int64_t B, int64_t L) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b < B) first_reject[b] = static_cast<int32_t>(L);
}

// Arg-max of one row: lowest id among the largest values (NaN below -inf).
__device__ int32_t row_argmax(VerifySmem& s, const uint16_t* row, int64_t V) {
  const int64_t nvec = V >> 3;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  uint64_t best = 0ull;   // (order << 32) | ~id
  int64_t i = threadIdx.x;
  for (; i + 3 * kVThreads < nvec; i += 4 * kVThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ldg_stream(rv + i + u * kVThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t vo = bf16_order(vec_max_bits(v[u]));
      if (vo >= static_cast<uint32_t>(best >> 32)) {
        const uint32_t id0 = static_cast<uint32_t>((i + u * kVThreads) * 8);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t key = (static_cast<uint64_t>(bf16_order(lane_bits(v[u], k))) << 32) |
                               static_cast<uint64_t>(~(id0 + k));
          best = kmax(best, key);
        }
      }
    }
  }
  for (; i < nvec; i += kVThreads) {
    const uint4 v = ldg_stream(rv + i);
    const uint32_t id0 = static_cast<uint32_t>(i * 8);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      best = kmax(best, (static_cast<uint64_t>(bf16_order(lane_bits(v, k))) << 32) |
                            static_cast<uint64_t>(~(id0 + k)));
  }
  for (int64_t e = nvec * 8 + threadIdx.x; e < V; e += kVThreads)
    best = kmax(best, (static_cast<uint64_t>(bf16_order(row[e])) << 32) |
                          static_cast<uint64_t>(~static_cast<uint32_t>(e)));
  const uint64_t r = block_max_key(s, best);
  return static_cast<int32_t>(~static_cast<uint32_t>(r));
}

// Softmax statistics of one row at inverse-temperature c = log2(e) / T:
// row_max = max_v l_v, row_z = sum_v 2^((l_v - row_max) c).
__device__ void row_softmax_stats(VerifySmem& s, const uint16_t* row, int64_t V, float c) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = V >> 3;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  // Per thread: running max m and sum acc of 2^((l - m) c); each 8-element
  // vector is summed in fp32 and added in fp64, so the row sum keeps ~1e-7
  // relative accuracy.
  float m = -INFINITY;
  double acc = 0.0;
  auto absorb = [&](const uint4& v) {
    const float vm = bf16_bits_to_float(vec_max_bits(v));
    if (vm > m) {
      acc *= static_cast<double>(fast_exp2((m - vm) * c));
      m = vm;
    }
    const float mc = m * c;
    float vs = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) vs += fast_exp2(fmaf(bf16_bits_to_float(lane_bits(v, k)), c, -mc));
    acc += static_cast<double>(vs);
  };
  int64_t i = threadIdx.x;
  for (; i + 3 * kVThreads < nvec; i += 4 * kVThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ldg_stream(rv + i + u * kVThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) absorb(v[u]);
  }
  for (; i < nvec; i += kVThreads) absorb(ldg_stream(rv + i));
  for (int64_t e = nvec * 8 + threadIdx.x; e < V; e += kVThreads) {
    const float x = bf16_bits_to_float(row[e]);
    if (x > m) {
      acc *= static_cast<double>(fast_exp2((m - x) * c));
      m = x;
    }
    acc += static_cast<double>(fast_exp2((x - m) * c));
  }
  // combine (m, acc) over the block; the sum is carried in fp64
  float wm = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, o));
  if (lane == 0) s.m[warp] = wm;
  __syncthreads();
  float M = s.m[0];
#pragma unroll
  for (int w = 1; w < kVWarps; ++w) M = fmaxf(M, s.m[w]);
  double z = (m == -INFINITY) ? 0.0 : acc * static_cast<double>(fast_exp2((m - M) * c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  if (lane == 0) s.z[warp] = z;
  __syncthreads();
  if (threadIdx.x == 0) {
    double Z = 0.0;
    for (int w = 0; w < kVWarps; ++w) Z += s.z[w];
    s.row_max = M;
    s.row_z = Z;
  }
  __syncthreads();
}

// Inverse-CDF draw in id order over weights w_v = 2^((l_v - M) c), except that the
// n_cand candidate ids in s.cand use the fp64 weights s.candr.  target_u in [0, 1).
__device__ int32_t row_draw(VerifySmem& s, const uint16_t* row, int64_t V, float c, int n_cand,
                            double target_u) {
  const int tid = threadIdx.x;
  const float M = s.row_max, mc = M * c;
  const int64_t per = (V + kVThreads - 1) / kVThreads;   // contiguous elements per thread
  const int64_t v0 = tid * per, v1 = (v0 + per < V) ? v0 + per : V;
  double part = 0.0;
  for (int64_t v = v0; v < v1; ++v) part += static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[v]), c, -mc)));
  for (int j = 0; j < n_cand; ++j) {
    const int64_t cv = s.cand[j];
    if (cv >= v0 && cv < v1)
      part += s.candr[j] - static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[cv]), c, -mc)));
  }
  part = part > 0.0 ? part : 0.0;
  // exclusive scan of the per-thread masses in thread (= id) order
  s.scan[tid] = part;
  __syncthreads();
  if (tid == 0) {
    double run = 0.0;
    for (int i = 0; i < kVThreads; ++i) {
      const double p = s.scan[i];
      s.scan[i] = run;
      run += p;
    }
    s.row_z = run;   // total residual mass (row_z is no longer needed)
    s.token = -1;
  }
  __syncthreads();
  const double total = s.row_z;
  const double target = target_u * total;
  const double lo = s.scan[tid];
  const double hi = (tid + 1 < kVThreads) ? s.scan[tid + 1] : total;
  if (lo <= target && target < hi && v1 > v0) {
    double run = lo;
    int32_t pick = -1, last_pos = -1;
    for (int64_t v = v0; v < v1; ++v) {
      double w = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[v]), c, -mc)));
      for (int j = 0; j < n_cand; ++j)
        if (s.cand[j] == v) w = s.candr[j];
      if (w > 0.0) last_pos = static_cast<int32_t>(v);
      run += w;
      if (target < run) {
        pick = static_cast<int32_t>(v);
        break;
      }
    }
    s.token = pick >= 0 ? pick : (last_pos >= 0 ? last_pos : static_cast<int32_t>(v0));
  }
  __syncthreads();
  return s.token;
}

__global__ void __launch_bounds__(kVThreads)
    verify_rows_kernel(const uint16_t* __restrict__ target, int64_t ld,
                       const int32_t* __restrict__ draft_tok, const int32_t* __restrict__ draft_slot,
                       const float* __restrict__ draft_q, const int32_t* __restrict__ cand_idx,
                       int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                       uint64_t offset, int32_t* first_reject, int32_t* __restrict__ out_tok,
                       uint32_t* __restrict__ err) {
  __shared__ VerifySmem s;
  const int64_t t = blockIdx.x / B, b = blockIdx.x % B;
  if (threadIdx.x == 0) s.skip = (t > *reinterpret_cast<volatile int32_t*>(first_reject + b)) ? 1 : 0;
  __syncthreads();
  if (s.skip) return;
  const uint16_t* row = target + (b * (L + 1) + t) * ld;
  if (temperature <= 0.0f) {
    const int32_t a = row_argmax(s, row, V);
    if (threadIdx.x == 0) {
      out_tok[b * (L + 1) + t] = a;
      if (t < L && draft_tok[b * L + t] != a) atomicMin(first_reject + b, static_cast<int32_t>(t));
    }
    return;
  }
  const float c = kLog2e / temperature;
  row_softmax_stats(s, row, V, c);
  if (t == L) {
    const double u = philox_uniform24(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(L), 2, offset);
    const int32_t tok = row_draw(s, row, V, c, 0, u);
    if (threadIdx.x == 0) out_tok[b * (L + 1) + L] = tok;
    return;
  }
  // accept test: u1 q(x) Z < 2^((l_x - M) c)
  if (threadIdx.x == 0) {
    const int32_t x = clamp_token(draft_tok[b * L + t], V, err);
    int32_t slot = draft_slot[b * L + t];
    if (slot < 0 || slot >= kTopK) {
      raise_error(err, DFLASH2_DEVERR_BAD_SLOT);
      slot = slot < 0 ? 0 : kTopK - 1;
    }
    const double q = static_cast<double>(draft_q[(b * L + t) * kTopK + slot]);
    const double ex = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[x]), c, -s.row_max * c)));
    const double u1 = philox_uniform24(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 1, offset);
    s.skip = (u1 * q * s.row_z < ex) ? 1 : 0;   // 1 = accepted
  }
  if (threadIdx.x < kTopK) {
    const float mc = s.row_max * c;
    const int32_t cv = clamp_token(cand_idx[(b * L + t) * kTopK + threadIdx.x], V, err);
    const double e = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[cv]), c, -mc)));
    const double qz = static_cast<double>(draft_q[(b * L + t) * kTopK + threadIdx.x]) * s.row_z;
    s.cand[threadIdx.x] = cv;
    s.candr[threadIdx.x] = e - qz > 0.0 ? e - qz : 0.0;
  }
  __syncthreads();
  if (s.skip) return;   // accepted: nothing more for this row
  if (threadIdx.x == 0) atomicMin(first_reject + b, static_cast<int32_t>(t));
  const double u2 = philox_uniform24(seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 2, offset);
  const int32_t tok = row_draw(s, row, V, c, kTopK, u2);
  if (threadIdx.x == 0) out_tok[b * (L + 1) + t] = tok;
}

__global__ void verify_finalize_kernel(const int32_t* __restrict__ draft_tok, int64_t B, int64_t L,
                                       int32_t* accept_len, int32_t* __restrict__ out_tok) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int32_t n = accept_len[b];
  for (int64_t t = 0; t <= L; ++t) {
    if (t < n) out_tok[b * (L + 1) + t] = draft_tok[b * L + t];
    else if (t > n) out_tok[b * (L + 1) + t] = -1;
  }
  accept_len[b] = n + 1;
}

}  // namespace

cudaError_t launch_verify(const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                          const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                          int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                          uint64_t offset, int32_t* accept_len, int32_t* out_tok, uint32_t* err,
                          int num_sms, cudaStream_t stream) {
  (void)num_sms;
  const unsigned small_grid = static_cast<unsigned>((B + 255) / 256);
  verify_init_kernel<<<small_grid, 256, 0, stream>>>(accept_len, B, L);
  const int64_t rows = B * (L + 1);
  if (rows > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  verify_rows_kernel<<<static_cast<unsigned>(rows), kVThreads, 0, stream>>>(
      target, ld, draft_tok, draft_slot, draft_q, cand_idx, B, L, V, temperature, seed, offset,
      accept_len, out_tok, err);
  verify_finalize_kernel<<<small_grid, 256, 0, stream>>>(draft_tok, B, L, accept_len, out_tok);
  return cudaGetLastError();
}

}  // namespace dflash2
