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
  double cand_z;
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

// True once an earlier position of the sequence is known to reject, i.e. row t
// can no longer matter (first_reject only ever decreases).
__device__ __forceinline__ bool row_irrelevant(const int32_t* first_reject, int64_t t) {
  return t > *reinterpret_cast<const volatile int32_t*>(first_reject);
}

// Each warp polls first_reject every kPoll outer iterations and stops streaming
// when the row has become irrelevant; its partial result is then garbage, which
// is harmless because nothing derived from an irrelevant row is written.
constexpr int kPoll = 2;

__device__ __forceinline__ bool warp_should_stop(const int32_t* first_reject, int64_t t, int it) {
  if ((it % kPoll) != kPoll - 1) return false;
  int stop = 0;
  if ((threadIdx.x & 31) == 0) stop = row_irrelevant(first_reject, t) ? 1 : 0;
  return __shfl_sync(0xFFFFFFFFu, stop, 0) != 0;
}

// Arg-max of one row: lowest id among the largest values (NaN below -inf).
__device__ int32_t row_argmax(VerifySmem& s, const uint16_t* row, int64_t V, const int32_t* first_reject,
                              int64_t t) {
  const int64_t nvec = V >> 3;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  uint64_t best = 0ull;   // (order << 32) | ~id
  int64_t i = threadIdx.x;
  for (int it = 0; i + 3 * kVThreads < nvec; i += 4 * kVThreads, ++it) {
    if (warp_should_stop(first_reject, t, it)) {
      i = nvec;
      break;
    }
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ldg_stream(rv + i + u * kVThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // a vector only matters if its max beats the thread's best so far (a tie
      // with it has a larger id, and ids increase along the thread's stripe)
      const uint32_t vo = bf16_order(vec_max_bits(v[u]));
      if (vo > static_cast<uint32_t>(best >> 32)) {
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
  // an all-NaN row never sets a key: its arg-max is the lowest id, 0
  return r == 0ull ? 0 : static_cast<int32_t>(~static_cast<uint32_t>(r));
}

// Softmax statistics of one row at inverse-temperature c = log2(e) / T:
// row_max = max_v l_v, row_z = sum_v 2^((l_v - row_max) c).
__device__ void row_softmax_stats(VerifySmem& s, const uint16_t* row, int64_t V, float c,
                                  const int32_t* first_reject, int64_t t) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nvec = V >> 3;
  const uint4* rv = reinterpret_cast<const uint4*>(row);
  // Per thread: running max m and sum acc of 2^((l - m) c); each 8-element
  // vector is summed in fp32 and added with Kahan compensation (fp64 is slow on
  // this part), so the row sum keeps ~1e-7 relative accuracy.
  float m = -INFINITY;
  float acc = 0.0f, comp = 0.0f;
  auto add = [&](float x) {
    const float y = x - comp;
    const float t2 = acc + y;
    comp = (t2 - acc) - y;
    acc = t2;
  };
  auto absorb = [&](const uint4& v) {
    const float vm = bf16_bits_to_float(vec_max_bits(v));
    if (vm > m) {
      const float r = fast_exp2((m - vm) * c);
      acc *= r;
      comp *= r;
      m = vm;
    }
    const float mc = m * c;
    float vs = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) vs += fast_exp2(fmaf(bf16_bits_to_float(lane_bits(v, k)), c, -mc));
    add(vs);
  };
  int64_t i = threadIdx.x;
  for (int it = 0; i + 3 * kVThreads < nvec; i += 4 * kVThreads, ++it) {
    if (warp_should_stop(first_reject, t, it)) {
      i = nvec;
      break;
    }
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
      const float r = fast_exp2((m - x) * c);
      acc *= r;
      comp *= r;
      m = x;
    }
    add(fast_exp2((x - m) * c));
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
  double z = (m == -INFINITY) ? 0.0
                              : (static_cast<double>(acc) - static_cast<double>(comp)) *
                                    static_cast<double>(fast_exp2((m - M) * c));
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

__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// Inverse-CDF draw in id order over weights w_v = 2^((l_v - M) c), except that the
// n_cand candidate ids in s.cand use the fp64 weights s.candr.  target_u in [0, 1).
// Two levels, all loads coalesced: the row is cut into kVThreads contiguous
// tiles of `per` elements; each warp sums 32 tiles (lanes read consecutive
// 16-byte vectors, fp64 warp sum), candidates are corrected with shared-memory
// atomics, thread 0 forms the tile prefix and picks the tile holding the target
// mass, and warp 0 scans that tile 256 elements at a time (fp64 warp scan).
__device__ int32_t row_draw(VerifySmem& s, const uint16_t* row, int64_t V, float c, int n_cand,
                            double target_u) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float mc = s.row_max * c;
  const int64_t per = (((V + kVThreads - 1) / kVThreads) + 7) & ~int64_t(7);
  auto weight = [&](int64_t v) -> double {
    return static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[v]), c, -mc)));
  };
  for (int j = warp * 32; j < warp * 32 + 32; ++j) {
    const int64_t v0 = j * per, v1 = (v0 + per < V) ? v0 + per : V;
    double part = 0.0;
    for (int64_t v = v0 + lane * 8; v < v1; v += 256) {
      if (v + 8 <= v1) {
        const uint4 x = *reinterpret_cast<const uint4*>(row + v);
        float vs = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) vs += fast_exp2(fmaf(bf16_bits_to_float(lane_bits(x, k)), c, -mc));
        part += static_cast<double>(vs);
      } else {
        for (int64_t e = v; e < v1; ++e) part += weight(e);
      }
    }
    part = warp_sum_f64(part);
    if (lane == 0) s.scan[j] = part;
  }
  __syncthreads();
  if (tid < n_cand) atomicAdd(&s.scan[s.cand[tid] / per], s.candr[tid] - weight(s.cand[tid]));
  __syncthreads();
  if (tid == 0) {
    double run = 0.0, target = 0.0;
    int pick = -1;
    double total = 0.0;
    for (int j = 0; j < kVThreads; ++j) total += (s.scan[j] > 0.0 ? s.scan[j] : 0.0);
    target = target_u * total;
    for (int j = 0; j < kVThreads; ++j) {
      const double pj = s.scan[j] > 0.0 ? s.scan[j] : 0.0;
      if (pj > 0.0) {
        if (target < run + pj || pick < 0) {
          pick = j;
          s.row_z = run;            // mass before the picked tile
        }
        if (target < run + pj) break;
      }
      run += pj;
    }
    s.token = pick;
    s.cand_z = target;
  }
  __syncthreads();
  const int tile = s.token;
  __syncthreads();
  if (warp == 0) {
    int32_t found = -1, last_pos = -1;
    if (tile >= 0) {
      const double target = s.cand_z;
      double base = s.row_z;
      const int64_t v0 = tile * per, v1 = (v0 + per < V) ? v0 + per : V;
      for (int64_t cbase = v0; cbase < v1 && found < 0; cbase += 256) {
        const int64_t v = cbase + lane * 8;
        double w[8];
        double mine = 0.0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          w[k] = 0.0;
          if (v + k < v1) {
            w[k] = weight(v + k);
            for (int j = 0; j < n_cand; ++j)
              if (s.cand[j] == v + k) w[k] = s.candr[j];
          }
          mine += w[k];
        }
        // inclusive warp scan of the lane masses
        double incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const double chunk = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, target < base + incl);
        int lp = -1;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (w[k] > 0.0) lp = static_cast<int>(v + k);
        const unsigned has = __ballot_sync(0xFFFFFFFFu, lp >= 0);
        if (has) last_pos = __shfl_sync(0xFFFFFFFFu, lp, 31 - __clz(has));
        if (hit) {
          const int src = __ffs(hit) - 1;
          int32_t pick = -1;
          if (lane == src) {
            double run = base + incl - mine;
            for (int k = 0; k < 8 && pick < 0; ++k) {
              run += w[k];
              if (target < run && w[k] > 0.0) pick = static_cast<int32_t>(v + k);
            }
            if (pick < 0) pick = lp;
          }
          found = __shfl_sync(0xFFFFFFFFu, pick, src);
        }
        base += chunk;
      }
    }
    if (lane == 0) s.token = found >= 0 ? found : (last_pos >= 0 ? last_pos : 0);
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
    const int32_t a = row_argmax(s, row, V, first_reject + b, t);
    if (threadIdx.x == 0 && !row_irrelevant(first_reject + b, t)) {
      out_tok[b * (L + 1) + t] = a;
      if (t < L && draft_tok[b * L + t] != a) atomicMin(first_reject + b, static_cast<int32_t>(t));
    }
    return;
  }
  const float c = kLog2e / temperature;
  row_softmax_stats(s, row, V, c, first_reject + b, t);
  if (threadIdx.x == 0) s.skip = row_irrelevant(first_reject + b, t) ? 1 : 0;
  __syncthreads();
  if (s.skip) return;
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
