// verify.cu -- block verification against the target's logits ("DFlash 2: Keep
// Drafting Parallel": the target checks the whole block in one forward pass;
// "A Lightweight Path Selector": rejection sampling restores the exact target
// distribution; Table 1's note: the acceptance length includes the verifier's
// next token).
//
// Row t of a sequence only matters while every earlier position accepted.  One
// cooperative launch (all CTAs resident) reads the rows position-major: each
// target row is cut into contiguous chunks of about 4096 ids, one warp's item,
// and the (t, chunk, b) items are strided over all warps of the grid in that
// order (sequences fastest, so that each sequence's work is spread over SMs).  A row is dead once an earlier position of its sequence is known to
// have rejected (first_reject only falls, so a dead row stays dead); a warp
// checks its next 32 items at once, with the loads of the first already in
// flight, and skips the dead ones.  Rows within about one position of the
// decided front are read in vain.
//   T = 0: the row's arg-max key (value order, then lowest id) is kept by a
//          64-bit atomic max per row; a chunk holding a key above the draft
//          token's rejects the row at once (atomicMin on first_reject), so no
//          chunk waits for another.  After a grid barrier, row n's key gives
//          its token.
//   T > 0: each chunk leaves its max and sum of 2^((l - max) c), c = log2(e) / T,
//          in scratch; the warp that completes a row's last chunk combines them
//          and tests u1 q(x) Z < 2^((l_x - M) c); a rejection lowers
//          first_reject[b].  After a grid barrier each sequence draws the token
//          of row n = first_reject[b]: from the residual max(0, e_v - q_v Z)
//          after a rejection, from p itself for the bonus row n = L; in id
//          order, the chunk by its mass, then inside the chunk (re-read) a run
//          of vectors, a vector and an id.
// After a last barrier: out_tok = draft[0..n-1], row n's token, -1...;
// accept_len[b] = n + 1.  Every barrier wait is bounded (2 s, then
// DFLASH2_DEVERR_TIMEOUT and every CTA stops).
#include "common.cuh"
#include "launch.h"
#include "philox.cuh"

namespace dflash2 {
namespace {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVUnroll = 8;          // 16-byte loads in flight per lane
constexpr int kChunkIds = 4096;      // target ids per chunk (one warp's item)
constexpr int kVCtasPerSm = 4;          // T = 0 (64 registers)
constexpr int kVCtasPerSmSampled = 3;   // T > 0 (85 registers)
constexpr int kDrawVecs = 5120;      // largest chunk a draw handles: 40960 ids
constexpr int kMaxChunks = kVThreads; // chunks per row the draws combine in one step (V < 10.5M)
constexpr float kLog2e = 1.4426950408889634f;

struct alignas(16) ChunkPartial {
  float m;          // the chunk's largest logit
  uint32_t pad;
  double z;         // sum over the chunk of 2^((l - m) c)
};

// Chunks per row (about kChunkIds ids each, at most kMaxChunks) and ids per
// chunk (a multiple of 8, at most kDrawVecs vectors while V < 10.5M).
__host__ __device__ inline int verify_chunks(int64_t V) {
  int64_t n = (V + kChunkIds - 1) / kChunkIds;
  if (n < 1) n = 1;
  if (n > kMaxChunks) n = kMaxChunks;
  return static_cast<int>(n);
}
__host__ __device__ inline int64_t verify_chunk_ids(int64_t V) {
  const int n = verify_chunks(V);
  return (((V + n - 1) / n) + 7) & ~int64_t(7);
}

// scratch layout: barrier words | arrival counters [rows] | row keys [rows] | partials [rows, chunks]
struct ScratchLayout {
  size_t counters, keys, partials, total;
  __host__ __device__ ScratchLayout(int64_t rows, int nch) {
    counters = 256;
    keys = counters + ((static_cast<size_t>(rows) * 4 + 255) / 256) * 256;
    partials = keys + ((static_cast<size_t>(rows) * 8 + 255) / 256) * 256;
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
  int abort;
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
  float vmass[kDrawVecs];     // draw: mass of each 8-id vector of the chunk
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = kmax(k, __shfl_xor_sync(0xFFFFFFFFu, k, o));
  return k;
}

__device__ __forceinline__ float warp_max_f32(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
  return x;
}

// An id's key: (value order << 32) | ~id, so that the largest key is the
// largest value and, among equal values, the lowest id; NaN orders below -inf
// (ranked among themselves by id), -0 equals +0.
__device__ __forceinline__ uint64_t id_key(uint32_t bits, uint32_t id) {
  return (static_cast<uint64_t>(bf16_order(bits)) << 32) | static_cast<uint64_t>(~id);
}

// ---------------------------------------------------------------------------
// one chunk [v0, v1) of a row (v0 % 8 == 0), one warp
// ---------------------------------------------------------------------------
// The chunk's vectors are read in batches of U per lane (lane + 32 u, in
// increasing order per lane).  The caller issues the first batch (load_batch)
// before it knows whether the item is live, so that the check's loads and the
// data's are in flight together.
template <int U>
__device__ __forceinline__ void load_batch(uint4 (&v)[U], const uint4* rv, int base, int nvec, int lane) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = base + lane + 32 * u;
    v[u] = i < nvec ? ldg_stream(rv + i) : make_uint4(0, 0, 0, 0);
  }
}

// Largest key of the chunk.  Each lane keeps its best vector maximum, the
// first vector holding it (a lane's first vector starts as best even if all
// NaN) and that vector's data, then names the lowest id with that value; the
// warp takes the largest key.  0 only for an empty chunk.  Per batch the lane
// first takes the batch maximum (a tree over the vectors' maxima); only a
// batch that beats the lane's best (the first, as a rule, then rarely) looks
// for its first vector holding that maximum.  v holds the first batch on entry.
template <int U>
__device__ __forceinline__ uint64_t warp_chunk_argmax(uint4 (&v)[U], const uint4* rv, int64_t v0, int64_t v1,
                                                      const uint16_t* row, int lane) {
  const int nvec = static_cast<int>((v1 - v0) >> 3);
  uint32_t best = 0u;
  int best_i = -1;
  uint4 bestv = make_uint4(0, 0, 0, 0);
  for (int base = 0;;) {
    uint32_t vm[U];
#pragma unroll
    for (int u = 0; u < U; ++u) vm[u] = base + lane + 32 * u < nvec ? vec_max_bits(v[u]) : 0x7FC0u;   // NaN: never a maximum
    uint32_t bm = vm[0];
#pragma unroll
    for (int u = 1; u < U; ++u) {
      const __nv_bfloat16 m = __hmax(__ushort_as_bfloat16(static_cast<unsigned short>(bm)),
                                     __ushort_as_bfloat16(static_cast<unsigned short>(vm[u])));
      bm = __bfloat16_as_ushort(m);
    }
    if (base + lane < nvec) {
      const uint32_t bo = bf16_order(bm);
      if (best_i < 0 || bo > best) {
        // the batch's first vector holding its maximum (its first vector if all NaN)
        const float bf = bf16_bits_to_float(bm);
        int pick = 0;
        uint4 pv = v[0];
#pragma unroll
        for (int u = U - 1; u >= 0; --u) {
          if (base + lane + 32 * u < nvec && bf16_bits_to_float(vm[u]) == bf) {
            pick = u;
            pv = v[u];
          }
        }
        best = bo;
        best_i = base + lane + 32 * pick;
        bestv = pv;
      }
    }
    base += 32 * U;
    if (base >= nvec) break;
    load_batch<U>(v, rv, base, nvec, lane);
  }
  uint64_t key = 0ull;
  if (best_i >= 0) {
    const uint32_t id0 = static_cast<uint32_t>(v0 + static_cast<int64_t>(best_i) * 8);
#pragma unroll
    for (int k = 0; k < 8; ++k) key = kmax(key, id_key(lane_bits(bestv, k), id0 + k));
  }
  for (int64_t e = v0 + static_cast<int64_t>(nvec) * 8 + lane; e < v1; e += 32)
    key = kmax(key, id_key(row[e], static_cast<uint32_t>(e)));
  return warp_max_u64(key);
}

// Softmax statistics of the chunk at inverse temperature c: its max m and
// z = sum 2^((l - m) c).  Per lane a running max and a Kahan-compensated fp32
// sum of per-vector fp32 sums (~1e-7 relative); the warp combines in fp64.
// Every lane returns m and z.  v holds the first batch on entry.
template <int U>
__device__ __forceinline__ void warp_chunk_stats(uint4 (&v)[U], const uint4* rv, int64_t v0, int64_t v1, const uint16_t* row,
                                 float c, int lane, float* m_out, double* z_out) {
  const int nvec = static_cast<int>((v1 - v0) >> 3);
  float m = -INFINITY;
  float acc = 0.0f, comp = 0.0f;
  auto add = [&](float x) {
    const float y = x - comp;
    const float t2 = acc + y;
    comp = (t2 - acc) - y;
    acc = t2;
  };
  auto rescale = [&](float nm) {
    const float r = fast_exp2((m - nm) * c);
    acc *= r;
    comp *= r;
    m = nm;
  };
  for (int base = 0;;) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + lane + 32 * u < nvec) {
        const float vm = bf16_bits_to_float(vec_max_bits(v[u]));
        if (vm > m) rescale(vm);
        const float mc = m * c;
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = fast_exp2(fmaf(bf16_bits_to_float(lane_bits(v[u], k)), c, -mc));
        add(((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7])));
      }
    }
    base += 32 * U;
    if (base >= nvec) break;
    load_batch<U>(v, rv, base, nvec, lane);
  }
  for (int64_t e = v0 + static_cast<int64_t>(nvec) * 8 + lane; e < v1; e += 32) {
    const float x = bf16_bits_to_float(row[e]);
    if (x > m) rescale(x);
    add(fast_exp2((x - m) * c));
  }
  const float M = warp_max_f32(m);
  double z = (m == -INFINITY) ? 0.0
                              : (static_cast<double>(acc) - static_cast<double>(comp)) *
                                    static_cast<double>(fast_exp2((m - M) * c));
  *m_out = M;
  *z_out = warp_sum_f64(z);
}


// Inclusive fp64 prefix sum over the warp's lanes (every lane calls).
__device__ __forceinline__ double warp_scan_incl(double x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Inverse-CDF pick over lanes in order, lane j holding mass w_j >= 0 and
// incl_j = sum_{i <= j} w_i: the first lane with w > 0 whose inclusive mass
// passes target, else (rounding) the last lane with w > 0, else -1.  *before
// gets the picked lane's exclusive prefix (0 if none).  Every lane calls.
__device__ __forceinline__ int warp_pick(double w, double incl, double target, int lane, double* before) {
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, w > 0.0 && target < incl);
  const unsigned pos = __ballot_sync(0xFFFFFFFFu, w > 0.0);
  const int src = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
  double excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) excl = 0.0;
  const double b = __shfl_sync(0xFFFFFFFFu, excl, src < 0 ? 0 : src);
  *before = src < 0 ? 0.0 : b;
  return src;
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
    // the run's vectors (lane j: vector pick * per + j), then the picked
    // vector's ids (lane k: id a + k, a candidate at its residual); without a
    // hit (rounding) the last vector and id of positive weight
    int32_t token = static_cast<int32_t>(v0);
    if (pick >= 0) {
      const double tgt = target - before;
      const int i = pick * per + lane;
      const double m = lane < per && i < nv ? static_cast<double>(fmaxf(s.vmass[i], 0.0f)) : 0.0;
      double vec_base;
      const int vj = warp_pick(m, warp_scan_incl(m, lane), tgt, lane, &vec_base);
      if (vj >= 0) {
        const int64_t id = v0 + static_cast<int64_t>(pick * per + vj) * 8 + lane;
        double w = 0.0;
        if (lane < 8 && id < v1) {
          w = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(row[id]), c, -mc)));
          for (int q = 0; q < n_cand; ++q)
            if (s.cand[q] == id) w = s.candr[q];
        }
        const double incl_w = warp_scan_incl(w, lane);
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, w > 0.0 && tgt < vec_base + incl_w);
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, w > 0.0);
        if (hit) token = static_cast<int32_t>(v0 + static_cast<int64_t>(pick * per + vj) * 8 + __ffs(hit) - 1);
        else if (pos) token = static_cast<int32_t>(v0 + static_cast<int64_t>(pick * per + vj) * 8 + 31 - __clz(pos));
      }
    }
    if (lane == 0) s.token = token;
  }
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
__global__ void verify_init_kernel(int32_t* first_reject, uint32_t* counters, unsigned long long* keys, unsigned* bar,
                                   int64_t B, int64_t L) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = B * (L + 1);
  if (i < B) first_reject[i] = static_cast<int32_t>(L);
  if (i < rows) {
    counters[i] = 0u;
    keys[i] = 0ull;
  }
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
  uint32_t* counters;      // T > 0: chunks completed per row
  unsigned long long* keys;   // T = 0: the row's largest key
  ChunkPartial* partials;  // T > 0: [rows, chunks]
  unsigned* bar;           // [0] count, [1] generation, [2] abort
  uint32_t* err;
};

// T > 0, the warp that completed row (b, t): the row's max M and Z from its
// chunk partials (lane q reads chunks q, q + 32, ...; fixed order, fp64), then
// the accept test u1 q(x) Z < 2^((l_x - M) c); a rejection lowers first_reject[b].
__device__ void decide_sampled_row(const VerifyArgs& a, const ChunkPartial* part, int nch, const uint16_t* row,
                                   int64_t b, int64_t t, float c, int lane) {
  const int64_t L = a.L;
  if (t >= L) return;   // the bonus row has no test
  int32_t f = 0;
  if (lane == 0) f = *reinterpret_cast<volatile int32_t*>(a.first_reject + b);
  if (t > __shfl_sync(0xFFFFFFFFu, f, 0)) return;   // past a known rejection (warp-uniform)
  uint32_t lx = 0u;
  int32_t slot = 0;
  if (lane == 0) {
    lx = row[clamp_token(a.draft_tok[b * L + t], a.V, a.err)];   // in flight with the partials
    slot = a.draft_slot[b * L + t];
  }
  constexpr int kPer = kMaxChunks / 32;
  float mq[kPer];
  double zq[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int q = lane + 32 * k;
    mq[k] = -INFINITY;
    zq[k] = 0.0;
    if (q < nch) {
      mq[k] = __ldcg(&part[q].m);
      zq[k] = __ldcg(&part[q].z);
    }
  }
  float ml = mq[0];
#pragma unroll
  for (int k = 1; k < kPer; ++k) ml = fmaxf(ml, mq[k]);
  const float M = warp_max_f32(ml);
  double zl = 0.0;
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (mq[k] != -INFINITY) zl += zq[k] * static_cast<double>(fast_exp2((mq[k] - M) * c));
  const double Z = warp_sum_f64(zl);
  if (lane == 0) {
    if (slot < 0 || slot >= kTopK) {
      raise_error(a.err, DFLASH2_DEVERR_BAD_SLOT);
      slot = slot < 0 ? 0 : kTopK - 1;
    }
    const double q = static_cast<double>(a.draft_q[(b * L + t) * kTopK + slot]);
    const double ex = static_cast<double>(fast_exp2(fmaf(bf16_bits_to_float(lx), c, -M * c)));
    const double u1 = philox_uniform24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 1, a.offset);
    if (!(u1 * q * Z < ex)) atomicMin(a.first_reject + b, static_cast<int32_t>(t));
  }
}

// A work item's (position, sequence, chunk).
struct ItemPos {
  int t, b, ch;
};

// p + d for d's components below their moduli (b < B, ch < nch): one carry each.
__device__ __forceinline__ ItemPos item_add(ItemPos p, ItemPos d, int nch, int B) {
  ItemPos r;
  r.b = p.b + d.b;
  const int c1 = r.b >= B;
  r.b -= c1 ? B : 0;
  r.ch = p.ch + d.ch + c1;
  const int c2 = r.ch >= nch;
  r.ch -= c2 ? nch : 0;
  r.t = p.t + d.t + c2;
  return r;
}

template <bool kSampled>
__global__ void __launch_bounds__(kVThreads, kSampled ? kVCtasPerSmSampled : kVCtasPerSm)
    verify_kernel(const VerifyArgs a) {
  __shared__ VerifySmem s;
  pdl_launch_dependents();   // launched in full order after its init kernel; lets the next kernel prepare
  const int64_t B = a.B, L = a.L, V = a.V;
  const int nch = verify_chunks(V);
  const int64_t cs = verify_chunk_ids(V);
  const float c = kSampled ? kLog2e / a.temperature : 0.0f;
  volatile int32_t* fr = a.first_reject;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s.abort = 0;
  __syncthreads();
  {
    // item = (t * nch + ch) * B + b: position-major, the sequence fastest, so a
    // sequence's chunks fall on warps of different CTAs (and SMs) and the work
    // of the sequences still alive stays spread over the GPU.  Positions are
    // stepped by carry-adds of precomputed (t, ch, b) offsets, so the loop
    // divides nothing.
    const int64_t per_pos = B * nch;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kVWarps;
    auto split = [&](int64_t x) {
      ItemPos p;
      p.t = static_cast<int>(x / per_pos);
      const int64_t r = x % per_pos;
      p.ch = static_cast<int>(r / B);
      p.b = static_cast<int>(r % B);
      return p;
    };
    const int Bi = static_cast<int>(B);
    const ItemPos stride = split(nwarps), ahead = split(lane * nwarps);
    ItemPos cur = split(static_cast<int64_t>(blockIdx.x) * kVWarps + (threadIdx.x >> 5));
    while (cur.t <= L) {
      const int t = cur.t, b = cur.b, ch = cur.ch;
      const int64_t ri = static_cast<int64_t>(b) * (L + 1) + t;
      const uint16_t* row = a.target + ri * a.ld;
      const int64_t v0 = ch * cs < V ? ch * cs : V, v1 = v0 + cs < V ? v0 + cs : V;
      const uint4* rv = reinterpret_cast<const uint4*>(row + v0);
      const int nvec = static_cast<int>((v1 - v0) >> 3);
      // the first batch, then (with it in flight) whether this item and the
      // warp's next 31 are live
      uint4 v[kVUnroll];
      load_batch<kVUnroll>(v, rv, 0, nvec, lane);
      int32_t dt = -1;
      uint32_t dbits = 0u;
      if (!kSampled && lane == 0 && t < L) {
        dt = a.draft_tok[static_cast<int64_t>(b) * L + t];
        if (dt >= 0 && dt < V) dbits = row[dt];
      }
      const ItemPos mine = item_add(cur, ahead, nch, Bi);
      const bool live = mine.t <= L && mine.t <= fr[mine.b];
      const unsigned mask = __ballot_sync(0xFFFFFFFFu, live);
      if (!(mask & 1u)) {
        // the first live one of the 32, else the one after them
        const int k = mask ? __ffs(mask) - 1 : 31;
        cur.t = __shfl_sync(0xFFFFFFFFu, mine.t, k);
        cur.b = __shfl_sync(0xFFFFFFFFu, mine.b, k);
        cur.ch = __shfl_sync(0xFFFFFFFFu, mine.ch, k);
        if (!mask) cur = item_add(cur, stride, nch, Bi);
        continue;
      }
      if (!kSampled) {
        const uint64_t key = warp_chunk_argmax<kVUnroll>(v, rv, v0, v1, row, lane);
        if (lane == 0) {
          if (key) atomicMax(a.keys + ri, static_cast<unsigned long long>(key));
          // a key above the draft token's rejects the row (an id outside [0, V)
          // is never the arg-max)
          if (t < L && (dt < 0 || dt >= V || key > id_key(dbits, static_cast<uint32_t>(dt))))
            atomicMin(a.first_reject + b, static_cast<int32_t>(t));
        }
      } else {
        float m;
        double z;
        warp_chunk_stats<kVUnroll>(v, rv, v0, v1, row, c, lane, &m, &z);
        ChunkPartial* part = a.partials + ri * nch;
        uint32_t prev = 0u;
        if (lane == 0) {
          part[ch].m = m;
          part[ch].z = z;
          __threadfence();
          prev = atomicAdd(a.counters + ri, 1u);
        }
        if (__shfl_sync(0xFFFFFFFFu, prev, 0) == static_cast<uint32_t>(nch - 1)) {
          __threadfence();
          decide_sampled_row(a, part, nch, row, b, t, c, lane);
        }
      }
      cur = item_add(cur, stride, nch, Bi);
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
      if (threadIdx.x < 32) {
        // warp 0: the chunk by its mass (inverse CDF in id order); lane j sums
        // chunks [j k, j k + k), the picked lane finds the chunk among its own
        const int k = (nch + 31) >> 5;
        double lsum = 0.0;
        for (int i = 0; i < k; ++i) {
          const int q = lane * k + i;
          if (q < nch) lsum += s.pmass[q] > 0.0 ? s.pmass[q] : 0.0;
        }
        const double incl = warp_scan_incl(lsum, lane);
        const double total_mass = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const double u2 = philox_uniform24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(n), 2, a.offset);
        const double tgt = u2 * total_mass;
        double lane_before;
        const int src = warp_pick(lsum, incl, tgt, lane, &lane_before);
        if (lane == (src < 0 ? 0 : src)) {
          double run = lane_before, before = 0.0;
          int pick = -1;
          for (int i = 0; src >= 0 && i < k; ++i) {
            const int q = lane * k + i;
            if (q >= nch) break;
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
      }
      __syncthreads();
      const int64_t d0 = s.pick * cs < V ? s.pick * cs : V, d1 = d0 + cs < V ? d0 + cs : V;
      const int32_t tok = chunk_draw(s, row, d0, d1, c, n_cand);
      // this sequence's outputs: the accepted prefix, row n's token, then -1
      for (int64_t t = threadIdx.x; t <= L; t += kVThreads)
        a.out_tok[b * (L + 1) + t] = t < n ? a.draft_tok[b * L + t] : (t == n ? tok : -1);
      __syncthreads();   // every thread has read first_reject[b]
      if (threadIdx.x == 0) a.first_reject[b] = static_cast<int32_t>(n + 1);
    }
    return;
  }
  if (kSampled) return;   // a barrier gave up: DFLASH2_DEVERR_TIMEOUT is raised
  // n = first_reject[b]: the accepted prefix, row n's token, then -1
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < B; b += stride) {
    const int32_t n = fr[b];
    for (int64_t t = 0; t <= L; ++t) {
      if (t < n) {
        a.out_tok[b * (L + 1) + t] = a.draft_tok[b * L + t];
      } else if (t == n) {
        if (!kSampled) {
          // row n's largest key (an all-NaN row's is its lowest id's, so 0 only if empty)
          const unsigned long long key = __ldcg(a.keys + b * (L + 1) + t);
          a.out_tok[b * (L + 1) + t] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key)) : 0;
        }
      } else {
        a.out_tok[b * (L + 1) + t] = -1;
      }
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
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(init_grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_init_kernel, accept_len,
                                             reinterpret_cast<uint32_t*>(sc + lay.counters),
                                             reinterpret_cast<unsigned long long*>(sc + lay.keys), bar, B, L);
    if (e != cudaSuccess) return e;
  }
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
  const int64_t ctas = ((L + 1) * B * nch + kVWarps - 1) / kVWarps;   // one warp per item at most
  const int grid = static_cast<int>(ctas < g ? ctas : g);
  VerifyArgs args{target, ld, draft_tok, draft_slot, draft_q, cand_idx, B, L, V, temperature, seed, offset,
                  accept_len, out_tok, reinterpret_cast<uint32_t*>(sc + lay.counters),
                  reinterpret_cast<unsigned long long*>(sc + lay.keys),
                  reinterpret_cast<ChunkPartial*>(sc + lay.partials), bar, err};
  void* kargs[] = {&args};
  return sampled ? cudaLaunchCooperativeKernel(reinterpret_cast<void*>(verify_kernel<true>), grid, kVThreads, kargs, 0,
                                               stream)
                 : cudaLaunchCooperativeKernel(reinterpret_cast<void*>(verify_kernel<false>), grid, kVThreads, kargs, 0,
                                               stream);
}

}  // namespace dflash2
