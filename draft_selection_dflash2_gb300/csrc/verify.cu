// verify.cu -- block verification against the target's logits ("DFlash 2: Keep
// Drafting Parallel": the target checks the whole block in one forward pass;
// "A Lightweight Path Selector": rejection sampling restores the exact target
// distribution; Table 1's note: the acceptance length includes the verifier's
// next token).
//
// Row t of a sequence only matters while every earlier position accepted.  One
// cooperative launch (all CTAs resident) reads the rows position-major: each
// target row is cut into contiguous chunks of ids, the (t, b, chunk) items are
// strided over the grid in that order, and an item is skipped once an earlier
// position of its sequence is known to have rejected, so only rows within
// about one position of the decided front are read in vain.  An item leaves its
// chunk's partial result in scratch:
//   T = 0: the largest key (value order, then lowest id);
//   T > 0: the chunk's max and sum of 2^((l - max) c), c = log2(e) / T.
// The CTA that completes a row's last chunk combines the partials and decides
// the row:
//   T = 0: out_tok := arg-max; a mismatch lowers first_reject[b] (atomicMin).
//   T > 0: accept iff u1 q(x) Z < 2^((l_x - M) c); a rejection lowers
//          first_reject[b].
// After a grid barrier, at T > 0, each sequence draws the token of row
// n = first_reject[b]: from the residual max(0, e_v - q_v Z) after a rejection,
// from p itself for the bonus row n = L; in id order, the chunk by its mass,
// then inside the chunk (re-read) a run of vectors, a vector and an id.  After a
// last barrier: out_tok = draft[0..n-1], row n's token, -1...; accept_len[b] =
// n + 1.  Every barrier wait is bounded (2 s, then DFLASH2_DEVERR_TIMEOUT and
// every CTA stops).
#include "common.cuh"
#include "launch.h"
#include "philox.cuh"

namespace dflash2 {
namespace {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVUnroll = 8;          // 16-byte loads in flight per thread
constexpr int kChunks = 4;           // chunks per target row (more if one would exceed kDrawVecs vectors)
constexpr int kVCtasPerSm = 4;          // T = 0 (64 registers)
constexpr int kVCtasPerSmSampled = 3;   // T > 0 (85 registers)
constexpr int kDrawVecs = 5120;      // largest chunk a draw handles: 40960 ids
constexpr int kMaxChunks = kVThreads; // chunks per row the decisions combine in one step (V < 10.5M)
constexpr float kLog2e = 1.4426950408889634f;

struct alignas(8) ChunkPartial {
  float m;          // T > 0: the chunk's largest logit
  uint32_t pad;
  double z;         // T > 0: sum over the chunk of 2^((l - m) c)
  uint64_t key;     // T = 0: (value order << 32) | ~id, 0 if the chunk is empty
};


// Chunks per row and ids per chunk (a multiple of 8, at most kDrawVecs vectors).
__host__ __device__ inline int verify_chunks(int64_t V) {
  const int64_t by_draw = (V + kDrawVecs * 8 - 1) / (kDrawVecs * 8);
  return static_cast<int>(by_draw > kChunks ? by_draw : kChunks);
}
__host__ __device__ inline int64_t verify_chunk_ids(int64_t V) {
  const int n = verify_chunks(V);
  return (((V + n - 1) / n) + 7) & ~int64_t(7);
}

// scratch layout: barrier words | arrival counters [rows] | partials [rows, chunks]
struct ScratchLayout {
  size_t counters, partials, total;
  __host__ __device__ ScratchLayout(int64_t rows, int nch) {
    counters = 256;
    partials = counters + ((static_cast<size_t>(rows) * 4 + 255) / 256) * 256;
    total = partials + static_cast<size_t>(rows) * nch * sizeof(ChunkPartial);
  }
};

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

__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

struct VerifySmem {
  int last, abort, skip[2];
  uint64_t key[kVWarps];
  float m[kVWarps];
  double z[kVWarps];
  // draws
  float row_max;
  double row_z;
  int pick, token;
  double target;              // mass still to pass inside the picked range
  int32_t cand[kTopK];
  double cande[kTopK];        // candidate weight 2^((l - M) c)
  double candr[kTopK];        // candidate residual max(0, e - q Z)
  double runs[kVThreads];     // draw: mass of each thread's run of vectors
  double pmass[kMaxChunks];   // the row's chunk masses relative to the row max
  uint32_t lx;                // accept test: the draft token's logit bits
  float vmass[kDrawVecs];     // draw: mass of each 8-id vector of the chunk
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
// one chunk [v0, v1) of a row (v0 % 8 == 0)
// ---------------------------------------------------------------------------
// Largest key of the chunk: (value order << 32) | ~id, so the lowest id wins ties.
// The stream keeps, per thread, only the best vector maximum and the first
// vector holding it (a strict > in the thread's increasing vector order keeps
// the first); the thread then re-reads that one vector to name the lowest id
// with that value.  NaN orders below -inf and never becomes a best (an all-NaN
// chunk gives key 0).
template <int U>
__device__ uint64_t chunk_argmax(const uint16_t* row, int64_t v0, int64_t v1) {
  const uint4* rv = reinterpret_cast<const uint4*>(row + v0);
  const int64_t nvec = (v1 - v0) >> 3;
  uint32_t best = 0u;       // value order of the best vector maximum (0: none yet)
  int64_t best_vec = -1;
  for (int64_t i = threadIdx.x; i < nvec; i += U * kVThreads) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = i + u * kVThreads < nvec ? ldg_stream(rv + i + u * kVThreads) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t vo = i + u * kVThreads < nvec ? bf16_order(vec_max_bits(v[u])) : 0u;
      const bool better = vo > best;
      best = better ? vo : best;
      best_vec = better ? i + u * kVThreads : best_vec;
    }
  }
  uint64_t key = 0ull;
  if (best_vec >= 0) {
    const uint4 v = rv[best_vec];
    const uint32_t id0 = static_cast<uint32_t>(v0 + best_vec * 8);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      key = kmax(key, (static_cast<uint64_t>(bf16_order(lane_bits(v, k))) << 32) | static_cast<uint64_t>(~(id0 + k)));
  }
  for (int64_t e = v0 + nvec * 8 + threadIdx.x; e < v1; e += kVThreads)
    key = kmax(key, (static_cast<uint64_t>(bf16_order(row[e])) << 32) |
                        static_cast<uint64_t>(~static_cast<uint32_t>(e)));
  return key;
}

// Softmax statistics of the chunk at inverse temperature c: its max m and
// z = sum 2^((l - m) c).  Per thread a running max and a Kahan-compensated fp32
// sum of per-vector fp32 sums (~1e-7 relative); the block combines in fp64.
template <int U>
__device__ void chunk_stats(VerifySmem& s, const uint16_t* row, int64_t v0, int64_t v1, float c, float* m_out,
                            double* z_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4* rv = reinterpret_cast<const uint4*>(row + v0);
  const int64_t nvec = (v1 - v0) >> 3;
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
  // every batch (the last, partial one included) has all its loads in flight at once
  for (int64_t i = threadIdx.x; i < nvec; i += U * kVThreads) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = i + u * kVThreads < nvec ? ldg_stream(rv + i + u * kVThreads) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (i + u * kVThreads >= nvec) break;
      absorb(v[u]);
    }
  }
  for (int64_t e = v0 + nvec * 8 + threadIdx.x; e < v1; e += kVThreads) {
    const float x = bf16_bits_to_float(row[e]);
    if (x > m) {
      const float r = fast_exp2((m - x) * c);
      acc *= r;
      comp *= r;
      m = x;
    }
    add(fast_exp2((x - m) * c));
  }
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
  z = warp_sum_f64(z);
  if (lane == 0) s.z[warp] = z;
  __syncthreads();
  if (threadIdx.x == 0) {
    double Z = 0.0;
    for (int w = 0; w < kVWarps; ++w) Z += s.z[w];
    *m_out = M;
    *z_out = Z;
  }
  __syncthreads();
}


// ---------------------------------------------------------------------------
// drawing inside one chunk
// ---------------------------------------------------------------------------
// Inverse-CDF draw over ids [v0, v1) (v0 % 8 == 0, at most kDrawVecs * 8 ids)
// with weights w_v = 2^((l_v - M) c), except that the n_cand candidates in
// s.cand weigh s.candr; the draw lands where the running mass first exceeds
// s.target.  One coalesced pass (loads four deep) leaves the fp32 mass of each
// 8-id vector in shared memory, candidates corrected; each thread sums a
// contiguous run of vectors (fp32, at most 20 terms), warp 0 scans the 256 run
// masses in fp64 and picks the run, and the run's owner picks the vector and
// the id.  Returns the id (the last id of positive weight if the target lies
// past the total, which only rounding can cause).
__device__ int32_t chunk_draw(VerifySmem& s, const uint16_t* row, int64_t v0, int64_t v1, float c, int n_cand) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float mc = s.row_max * c;
  const int nv = static_cast<int>((v1 - v0 + 7) >> 3);
  const uint4* rv = reinterpret_cast<const uint4*>(row + v0);
  auto weight = [&](int64_t v) -> float { return fast_exp2(fmaf(bf16_bits_to_float(row[v]), c, -mc)); };
#pragma unroll 4
  for (int i = tid; i < nv; i += kVThreads) {
    const int64_t v = v0 + static_cast<int64_t>(i) * 8;
    float w = 0.0f;
    if (v + 8 <= v1) {
      const uint4 x = ldg_stream(rv + i);
#pragma unroll
      for (int k = 0; k < 8; ++k) w += fast_exp2(fmaf(bf16_bits_to_float(lane_bits(x, k)), c, -mc));
    } else {
      for (int64_t e = v; e < v1; ++e) w += weight(e);
    }
    s.vmass[i] = w;
  }
  __syncthreads();
  if (tid < n_cand && s.cand[tid] >= v0 && s.cand[tid] < v1)
    atomicAdd(&s.vmass[(s.cand[tid] - v0) >> 3], static_cast<float>(s.candr[tid] - s.cande[tid]));
  __syncthreads();
  const int per = (nv + kVThreads - 1) / kVThreads;   // vectors per thread run
  {
    float part = 0.0f;
    for (int i = tid * per; i < nv && i < (tid + 1) * per; ++i) part += fmaxf(s.vmass[i], 0.0f);
    s.runs[tid] = static_cast<double>(part);
  }
  __syncthreads();
  if (tid < 32) {
    // warp 0: inclusive fp64 scan of the 256 run masses, 8 per lane
    double loc[8], acc = 0.0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc += s.runs[lane * 8 + k];
      loc[k] = acc;
    }
    double incl = acc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const double excl = incl - acc;
    const double target = s.target;
    // first run whose inclusive mass passes the target (runs of zero mass never win)
    int hit = -1;
#pragma unroll
    for (int k = 7; k >= 0; --k)
      if (s.runs[lane * 8 + k] > 0.0 && target < excl + loc[k]) hit = lane * 8 + k;
    const unsigned any = __ballot_sync(0xFFFFFFFFu, hit >= 0);
    int pick = -1;
    double before = 0.0;
    if (any) {
      const int src = __ffs(any) - 1;
      pick = __shfl_sync(0xFFFFFFFFu, hit, src);
    } else {
      // past the total: the last run of positive mass
      int lastp = -1;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (s.runs[lane * 8 + k] > 0.0) lastp = lane * 8 + k;
      const unsigned has = __ballot_sync(0xFFFFFFFFu, lastp >= 0);
      if (has) pick = __shfl_sync(0xFFFFFFFFu, lastp, 31 - __clz(has));
    }
    if (pick >= 0) {
      const int pl = pick >> 3, pk = pick & 7;
      double b = 0.0;
      double lk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) lk[k] = __shfl_sync(0xFFFFFFFFu, loc[k], pl);
      const double pe = __shfl_sync(0xFFFFFFFFu, excl, pl);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k == pk) b = pe + (k > 0 ? lk[k - 1] : 0.0);
      before = b;
    }
    if (lane == 0) {
      s.pick = pick;
      s.target = target - before;
    }
  }
  __syncthreads();
  if (tid == s.pick) {
    // the run's vectors, then the picked vector's ids (candidates at their residual);
    // without a hit (rounding) the last vector and id of positive weight
    double run = 0.0, vec_base = 0.0;
    int vec = -1;
    for (int i = tid * per; i < nv && i < (tid + 1) * per; ++i) {
      const double m = fmaxf(s.vmass[i], 0.0f);
      if (m > 0.0) {
        vec = i;
        vec_base = run;
        if (s.target < run + m) break;
      }
      run += m;
    }
    int32_t tok = -1, last_pos = -1;
    if (vec >= 0) {
      double r2 = vec_base;
      const int64_t a = v0 + static_cast<int64_t>(vec) * 8, e = a + 8 < v1 ? a + 8 : v1;
      const uint4 x = a + 8 <= v1 ? *reinterpret_cast<const uint4*>(row + a) : make_uint4(0, 0, 0, 0);
      for (int64_t v = a; v < e; ++v) {
        double w = a + 8 <= v1 ? static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(lane_bits(x, static_cast<int>(v - a))), c, -mc)))
                               : static_cast<double>(weight(v));
        for (int q = 0; q < n_cand; ++q)
          if (s.cand[q] == v) w = s.candr[q];
        if (w > 0.0) {
          last_pos = static_cast<int32_t>(v);
          r2 += w;
          if (tok < 0 && s.target < r2) tok = static_cast<int32_t>(v);
        }
      }
    }
    s.token = tok >= 0 ? tok : (last_pos >= 0 ? last_pos : static_cast<int32_t>(v0));
  }
  if (s.pick < 0 && tid == 0) s.token = static_cast<int32_t>(v0);
  __syncthreads();
  return s.token;
}


// T > 0: the row's max M and Z = sum 2^((l - M) c) from its chunk partials, all
// loads in parallel (thread q reads chunk q); leaves each chunk's mass relative
// to M in s.pmass.  Whole-CTA call.
__device__ void combine_row(VerifySmem& s, const ChunkPartial* part, int nch, float c) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mq = -INFINITY;
  double zq = 0.0;
  if (tid < nch) {
    mq = __ldcg(&part[tid].m);
    zq = __ldcg(&part[tid].z);
  }
  float wm = mq;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, o));
  if (lane == 0) s.m[warp] = wm;
  __syncthreads();
  float M = s.m[0];
#pragma unroll
  for (int w = 1; w < kVWarps; ++w) M = fmaxf(M, s.m[w]);
  const double mass = mq == -INFINITY ? 0.0 : zq * static_cast<double>(fast_exp2((mq - M) * c));
  if (tid < nch) s.pmass[tid] = mass;
  const double z = warp_sum_f64(mass);
  __syncthreads();
  if (lane == 0) s.z[warp] = z;
  __syncthreads();
  if (tid == 0) {
    double Z = 0.0;
    for (int w = 0; w < kVWarps; ++w) Z += s.z[w];
    s.row_max = M;
    s.row_z = Z;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// grid barrier (all CTAs are resident: cooperative launch)
// ---------------------------------------------------------------------------
// Sense by generation: the last CTA to arrive resets the count and bumps the
// generation.  A wait that passes kWaitLimitNs raises DFLASH2_DEVERR_TIMEOUT and
// sets the shared abort word, after which every CTA leaves its loops.
__device__ void grid_barrier(unsigned* count, volatile unsigned* gen, volatile unsigned* abort_word,
                             VerifySmem& s, uint32_t* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned g = *gen;
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      *count = 0u;
      __threadfence();
      *gen = g + 1;
    } else {
      const uint64_t start = global_timer_ns();
      while (*gen == g) {
        if (*abort_word) break;
        __nanosleep(64);
        if (global_timer_ns() - start > kWaitLimitNs) {
          raise_error(err, DFLASH2_DEVERR_TIMEOUT);
          *abort_word = 1u;
          break;
        }
      }
    }
    __threadfence();
    s.abort = *abort_word ? 1 : 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------
__global__ void verify_init_kernel(int32_t* first_reject, uint32_t* counters, unsigned* bar, int64_t B, int64_t L) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = B * (L + 1);
  if (i < B) first_reject[i] = static_cast<int32_t>(L);
  if (i < rows) counters[i] = 0u;
  if (i < 4) bar[i] = 0u;   // count, generation, abort
}

struct VerifyArgs {
  const uint16_t* target;
  int64_t ld;
  const int32_t* draft_tok;
  const int32_t* draft_slot;
  const float* draft_q;
  const int32_t* cand_idx;
  int64_t B, L, V;
  float temperature;
  uint64_t seed, offset;
  int32_t* first_reject;   // = accept_len until the end
  int32_t* out_tok;
  uint32_t* counters;
  ChunkPartial* partials;
  unsigned* bar;           // [0] count, [1] generation, [2] abort
  uint32_t* err;
};

template <bool kSampled>
__global__ void __launch_bounds__(kVThreads, kSampled ? kVCtasPerSmSampled : kVCtasPerSm)
    verify_kernel(const VerifyArgs a) {
  __shared__ VerifySmem s;
  const int64_t B = a.B, L = a.L, V = a.V;
  const int nch = verify_chunks(V);
  const int64_t cs = verify_chunk_ids(V);
  const float c = kSampled ? kLog2e / a.temperature : 0.0f;
  volatile int32_t* fr = a.first_reject;
  if (threadIdx.x == 0) s.abort = 0;
  __syncthreads();
  {
    const int64_t items = (L + 1) * B * nch;
    int parity = 0;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, parity ^= 1) {
      const int64_t t = item / (B * nch), b = (item / nch) % B;
      const int ch = static_cast<int>(item % nch);
      // a row past a known rejection is skipped; thread 0 decides for the whole CTA
      // (first_reject may change under it), through a slot that alternates with the
      // item so that one barrier suffices
      if (threadIdx.x == 0) s.skip[parity] = t > fr[b] ? 1 : 0;
      __syncthreads();
      if (s.skip[parity]) continue;
      const int64_t ri = b * (L + 1) + t;
      const uint16_t* row = a.target + ri * a.ld;
      const int64_t v0 = ch * cs < V ? ch * cs : V, v1 = v0 + cs < V ? v0 + cs : V;
      ChunkPartial* out = a.partials + ri * nch + ch;
      if (!kSampled) {
        const uint64_t key = block_max_key(s, chunk_argmax<kVUnroll>(row, v0, v1));
        if (threadIdx.x == 0) out->key = key;
      } else {
        float m;
        double z;
        chunk_stats<kVUnroll>(s, row, v0, v1, c, &m, &z);
        if (threadIdx.x == 0) {
          out->m = m;
          out->z = z;
        }
      }
      if (threadIdx.x == 0) {
        __threadfence();
        s.last = (atomicAdd(a.counters + ri, 1u) == static_cast<uint32_t>(nch - 1)) ? 1 : 0;
      }
      __syncthreads();
      if (!s.last) continue;
      // the row's last chunk: decide it
      const ChunkPartial* part = a.partials + ri * nch;
      __threadfence();
      if (!kSampled) {
        uint64_t key = 0ull;
        for (int q = threadIdx.x; q < nch; q += kVThreads)
          key = kmax(key, __ldcg(reinterpret_cast<const unsigned long long*>(&part[q].key)));
        key = block_max_key(s, key);
        if (threadIdx.x == 0) {
          // an all-NaN row never sets a key: its arg-max is the lowest id, 0
          const int32_t tok = key == 0ull ? 0 : static_cast<int32_t>(~static_cast<uint32_t>(key));
          a.out_tok[ri] = tok;
          if (t < L && a.draft_tok[b * L + t] != tok) atomicMin(a.first_reject + b, static_cast<int32_t>(t));
        }
        __syncthreads();
        continue;
      }
      if (threadIdx.x == kVThreads - 1 && t < L)
        s.lx = row[clamp_token(a.draft_tok[b * L + t], V, a.err)];   // in flight with the partials
      combine_row(s, part, nch, c);
      if (threadIdx.x == 0) {
        const float M = s.row_max;
        const double Z = s.row_z;
        if (t < L && t <= fr[b]) {
          // accept test: u1 q(x) Z < 2^((l_x - M) c)
          int32_t slot = a.draft_slot[b * L + t];
          if (slot < 0 || slot >= kTopK) {
            raise_error(a.err, DFLASH2_DEVERR_BAD_SLOT);
            slot = slot < 0 ? 0 : kTopK - 1;
          }
          const double q = static_cast<double>(a.draft_q[(b * L + t) * kTopK + slot]);
          const double ex = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(s.lx), c, -M * c)));
          const double u1 =
              philox_uniform24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 1, a.offset);
          if (!(u1 * q * Z < ex)) atomicMin(a.first_reject + b, static_cast<int32_t>(t));
        }
      }
      __syncthreads();
    }
    grid_barrier(a.bar, a.bar + 1, a.bar + 2, s, a.err);
  }
  if (kSampled && !s.abort) {
    // the token of row n = first_reject[b]: residual after a rejection, p itself for the bonus
    for (int64_t b = blockIdx.x; b < B; b += gridDim.x) {
      const int64_t n = fr[b];
      const int64_t ri = b * (L + 1) + n;
      const uint16_t* row = a.target + ri * a.ld;
      const ChunkPartial* part = a.partials + ri * nch;
      const int n_cand = n < L ? kTopK : 0;
      combine_row(s, part, nch, c);
      if (threadIdx.x < n_cand) {
        const float mc = s.row_max * c;
        const int32_t cv = clamp_token(a.cand_idx[(b * L + n) * kTopK + threadIdx.x], V, a.err);
        const double e = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[cv]), c, -mc)));
        const double qz = static_cast<double>(a.draft_q[(b * L + n) * kTopK + threadIdx.x]) * s.row_z;
        s.cand[threadIdx.x] = cv;
        s.cande[threadIdx.x] = e;
        s.candr[threadIdx.x] = e - qz > 0.0 ? e - qz : 0.0;
      }
      __syncthreads();
      if (threadIdx.x < n_cand) {
        // candidates' residual corrections of their chunks' masses
        const int q = static_cast<int>(s.cand[threadIdx.x] / cs);
        atomicAdd(&s.pmass[q], s.candr[threadIdx.x] - s.cande[threadIdx.x]);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        double total_mass = 0.0;
        for (int q = 0; q < nch; ++q) total_mass += s.pmass[q] > 0.0 ? s.pmass[q] : 0.0;
        const double u2 = philox_uniform24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(n), 2, a.offset);
        const double tgt = u2 * total_mass;
        double run = 0.0, before = 0.0;
        int pick = -1;
        for (int q = 0; q < nch; ++q) {
          const double pq = s.pmass[q] > 0.0 ? s.pmass[q] : 0.0;
          if (pq > 0.0) {
            pick = q;
            before = run;
            if (tgt < run + pq) break;
          }
          run += pq;
        }
        s.pick = pick < 0 ? 0 : pick;
        s.target = tgt - before;
      }
      __syncthreads();
      const int64_t d0 = s.pick * cs < V ? s.pick * cs : V, d1 = d0 + cs < V ? d0 + cs : V;
      const int32_t tok = chunk_draw(s, row, d0, d1, c, n_cand);
      if (threadIdx.x == 0) a.out_tok[ri] = tok;
      __syncthreads();
    }
    grid_barrier(a.bar, a.bar + 1, a.bar + 2, s, a.err);
  }
  // n = first_reject[b]: the accepted prefix, row n's token, then -1
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < B; b += stride) {
    const int32_t n = fr[b];
    for (int64_t t = 0; t <= L; ++t) {
      if (t < n) a.out_tok[b * (L + 1) + t] = a.draft_tok[b * L + t];
      else if (t > n) a.out_tok[b * (L + 1) + t] = -1;
    }
    a.first_reject[b] = n + 1;
  }
}

int max_verify_grid(bool sampled, int num_sms) {
  int per_sm = 0;
  const cudaError_t e = sampled ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<true>, kVThreads, 0)
                                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<false>, kVThreads, 0);
  if (e != cudaSuccess || per_sm < 1) return 0;
  return per_sm * num_sms;
}

}  // namespace

int64_t verify_max_vocab() { return static_cast<int64_t>(kMaxChunks) * kDrawVecs * 8; }

size_t verify_scratch_bytes(int64_t B, int64_t L, int64_t V) {
  return ScratchLayout(B * (L + 1), verify_chunks(V)).total;
}

cudaError_t launch_verify(const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                          const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                          int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                          uint64_t offset, int32_t* accept_len, int32_t* out_tok, void* scratch,
                          uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t rows = B * (L + 1);
  const int nch = verify_chunks(V);
  if (nch > kMaxChunks || rows > 0x7FFFFFFFLL / nch) return cudaErrorInvalidValue;
  const bool sampled = temperature > 0.0f;
  const ScratchLayout lay(rows, nch);
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  unsigned* bar = reinterpret_cast<unsigned*>(sc);
  const unsigned init_grid = static_cast<unsigned>((rows + 255) / 256);
  verify_init_kernel<<<init_grid, 256, 0, stream>>>(accept_len, reinterpret_cast<uint32_t*>(sc + lay.counters), bar,
                                                   B, L);
  // the co-resident grid, per device and variant
  static std::mutex mu;
  static int grid_cache[kMaxDevices][2] = {};
  int dev = 0;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int g;
  {
    std::lock_guard<std::mutex> lock(mu);
    int& cached = grid_cache[dev][sampled ? 1 : 0];
    if (cached == 0) cached = max_verify_grid(sampled, num_sms);
    g = cached;
  }
  if (g == 0) return cudaErrorInvalidConfiguration;
  const int64_t items = (L + 1) * B * nch;
  const int grid = static_cast<int>(items < g ? items : g);
  VerifyArgs args{target, ld, draft_tok, draft_slot, draft_q, cand_idx, B, L, V, temperature, seed, offset,
                  accept_len, out_tok, reinterpret_cast<uint32_t*>(sc + lay.counters),
                  reinterpret_cast<ChunkPartial*>(sc + lay.partials),
                  bar, err};
  void* kargs[] = {&args};
  return sampled ? cudaLaunchCooperativeKernel(reinterpret_cast<void*>(verify_kernel<true>), grid, kVThreads, kargs, 0,
                                               stream)
                 : cudaLaunchCooperativeKernel(reinterpret_cast<void*>(verify_kernel<false>), grid, kVThreads, kargs, 0,
                                               stream);
}

}  // namespace dflash2
