// verify.cu -- block verification against the target's logits ("DFlash 2: Keep
// Drafting Parallel": the target checks the whole block in one forward pass;
// "A Lightweight Path Selector": rejection sampling restores the exact target
// distribution; Table 1's note: the acceptance length includes the verifier's
// next token).
//
// Row t of a sequence only matters while every earlier position accepted
// (first_reject[b] only falls, so a row past it stays dead).  Rows are taken
// position-major, the sequence fastest.
//
// T = 0, one cooperative launch of the co-resident grid (no CTA waits for
//   another: the cooperative launch is kept for where it places the CTAs --
//   a plain launch of the same grid lands them on the SMs in another order and
//   measured 11% slower): each target row is cut into contiguous chunks of about
//   4096 ids, one warp's item, and the (t, chunk, b) items are strided over
//   all warps of the grid.  A warp checks its next 32 items' liveness at once,
//   with the loads of the first already in flight, and skips the dead ones.
//   The row's arg-max key (value order, then lowest id) is kept by a 64-bit
//   atomic max per row; a chunk holding a key above the draft token's rejects
//   the row at once (atomicMin on first_reject), so no chunk waits for
//   another.  The last CTA to finish (a counter raised after a fence) reads
//   row n's key for its token and writes the outputs; no CTA waits for another.
//
// T > 0, the target distribution in exact fixed point: with c = log2(e) / T
//   and M the row's largest non-NaN logit, every id weighs
//   W_v = floor(exp2_neg((l_v - M) c) 2^40), an integer, and p(v) = W_v / Z with
//   Z = sum_v W_v.  Integer sums are the same in any order, so partial sums
//   over slices give the exact Z and exact prefix sums.
//   verify_rows_kernel: one thread-block cluster of 8 CTAs per row.  Each CTA
//   copies its eighth of the row into shared memory with one bulk copy (TMA,
//   completing on an mbarrier; the next row's copy is requested once this
//   row is done), takes its maximum, and the 8 maxima meet in distributed
//   shared memory (cluster barrier); each CTA then sums its slice's weights
//   from shared memory, the 8 sums meet in CTA 0, which runs the accept test
//   (u1 q) Z < W_x in fp64, lowers first_reject[b] on a rejection and marks
//   the row decided.  A cluster takes a row only once the row before it in the
//   sequence is decided (a bounded wait on that flag), so nothing is read on
//   speculation.
//   verify_draw_kernel (one CTA per sequence): the token of row n =
//   first_reject[b] by inverse CDF in id order over integer prefix sums --
//   from the residual max(0, W_v - Q_v), Q_v = floor(q_v Z), after a rejection,
//   from W for the bonus row n = L -- with the target floor(U2 R / 2^24): the
//   slice by its mass, then inside it a thread's run of vectors, a vector and
//   an id, each level recomputed exactly.
// accept_len[b] = n + 1; out_tok = draft[0..n-1], row n's token, -1...
// Every wait is bounded (2 s, then DFLASH2_DEVERR_TIMEOUT).
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "philox.cuh"

namespace cg = cooperative_groups;

namespace dflash2 {
namespace {

// T = 0 pass
constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVUnroll = 8;          // 16-byte loads in flight per lane
constexpr int kChunkIds = 4096;      // target ids per chunk (one warp's item)
constexpr int kVCtasPerSm = 4;
constexpr int kMaxChunks = kVThreads;
// T > 0 passes
constexpr int kRowCluster = 8;       // CTAs per row
constexpr int kRowThreads = 256;
constexpr int kRowCtasPerSm = 4;
constexpr int kRowBuffers = 1;       // shared-memory piece buffers per CTA
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowWarpsC = kRowWarps;   // warp runs per slice (the draw reads their sums)
constexpr int kPieceIds = 20480;     // ids per shared-memory buffer (40 KB; a slice of V <= 163,840 fits one)
constexpr int kDrawThreads = 256;
constexpr int kDrawKeep = 2;         // run vectors a draw thread keeps in shared memory
constexpr float kLog2e = 1.44269504f;   // the walk's constant: the same fp32 value

// Chunks per row (about kChunkIds ids each, at most kMaxChunks) and ids per
// chunk (a multiple of 8).
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
// ids per CTA slice of a row (T > 0): an eighth, rounded up to a multiple of 8
// so that every slice starts on a 16-byte boundary
__host__ __device__ inline int64_t verify_slice_ids(int64_t V) {
  return (((V + kRowCluster - 1) / kRowCluster) + 7) & ~int64_t(7);
}

// workspace layout: barrier words | row values [rows] u64 (T = 0: arg-max key;
// T > 0: Z) | row maxima [rows] u32 (T > 0, order images) | decided flags
// [rows] u32 (T > 0) | slice sums [rows, 8] u64 (T > 0) | warp-run sums
// [rows, 8, warps] u64 (T > 0)
struct ScratchLayout {
  size_t rowval, rowmax, decided, slices, runs, total;
  __host__ __device__ explicit ScratchLayout(int64_t rows) {
    const size_t r = static_cast<size_t>(rows);
    rowval = 256;
    rowmax = rowval + ((r * 8 + 255) / 256) * 256;
    decided = rowmax + ((r * 4 + 255) / 256) * 256;
    slices = decided + ((r * 4 + 255) / 256) * 256;
    runs = slices + r * kRowCluster * 8;
    total = runs + r * kRowCluster * kRowWarpsC * 8;
  }
};

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
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

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = kmax(k, __shfl_xor_sync(0xFFFFFFFFu, k, o));
  return k;
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


// ---------------------------------------------------------------------------
// the fixed-point weights (T > 0)
// ---------------------------------------------------------------------------
// W = floor(exp2_neg(x) 2^40) with x = (l - M) c, taken in the steps of
// exp2_neg (exp2.cuh) but finished in the fixed point directly, with fp32
// operations only:
//   x <- max(x, -60): below -41 every weight floors to 0 on both paths, and
//        NaN (which exp2_neg maps to 0) becomes -60, which floors to 0 too;
//   n = rint(x) as t - 1.5 2^23 with t = x + 1.5 2^23, exact round-to-nearest-
//        even for |x| < 2^22, whose sum's low bits hold n;
//   f = x - n; p = the same degree-7 polynomial in the same Horner order;
//   y' = p 2^(n + 17) = exp2_neg(x) 2^40 / 2^23 exactly (2^(n+17) built from
//        t's bits; exp2_neg's own p 2^n is exact here, its result being normal);
//   a = floor(y') from t1 = y' + 2^23 rounded toward zero (y' < 2^18, so t1 has
//        integer resolution and holds 2^23 + a); frac = y' - a, exact;
//   b = floor(2^23 frac) from t2 = fma(frac, 2^23, 2^23) rounded toward zero;
//   W = 2^23 a + b, with a, b read from t1's and t2's bits minus 2^23's.
// Every step is a correctly rounded IEEE fp32 operation, so the integer is the
// same as the plain definition's on every input.
struct WeightParams {
  float M, c;
  __device__ WeightParams(float M_, float c_) : M(M_), c(c_) {}
};

__device__ __forceinline__ void fixed_weight_parts(float l, const WeightParams& wp, uint32_t& A, uint32_t& Bs) {
  float x = __fmul_rn(__fsub_rn(l, wp.M), wp.c);
  x = fmaxf(x, -60.0f);
  const float t = __fadd_rn(x, 12582912.0f);                 // 1.5 * 2^23 + n
  const float f = __fsub_rn(x, __fsub_rn(t, 12582912.0f));
  float p = 1.525273365e-05f;
  p = __fmaf_rn(p, f, 1.540352969e-04f);
  p = __fmaf_rn(p, f, 1.333355787e-03f);
  p = __fmaf_rn(p, f, 9.618128650e-03f);
  p = __fmaf_rn(p, f, 5.550410971e-02f);
  p = __fmaf_rn(p, f, 2.402265072e-01f);
  p = __fmaf_rn(p, f, 6.931471825e-01f);
  p = __fmaf_rn(p, f, 1.0f);
  // t's bits are 0x4B400000 + n; shifted by 23 they leave n in the exponent
  // field (0x4B400000's low 9 bits are 0), to which 127 + 17 is added
  const float yp = __fmul_rn(p, __uint_as_float((__float_as_uint(t) << 23) + (144u << 23)));
  const float t1 = __fadd_rz(yp, 8388608.0f);                // 2^23 + floor(y')
  const float fr = __fsub_rn(yp, __fsub_rn(t1, 8388608.0f));
  const float t2 = __fmaf_rz(fr, 8388608.0f, 8388608.0f);    // 2^23 + floor(2^23 frac)
  A += __float_as_uint(t1);
  Bs += __float_as_uint(t2);
}

// Packed fp32 pairs (Blackwell's f32x2 arithmetic: two independent fp32
// operations per instruction, each rounded exactly as the scalar operation
// with the same rounding mode).  Element 0 of a pair sits in the low 32 bits.
struct F2 {
  uint64_t v;
  __device__ __forceinline__ float lo() const { return __uint_as_float(static_cast<uint32_t>(v)); }
  __device__ __forceinline__ float hi() const { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
  return {static_cast<uint64_t>(__float_as_uint(hi)) << 32 | __float_as_uint(lo)};
}
__device__ __forceinline__ F2 f2_add_rn(F2 a, F2 b) {
  F2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}
__device__ __forceinline__ F2 f2_sub_rn(F2 a, F2 b) {
  F2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}
__device__ __forceinline__ F2 f2_mul_rn(F2 a, F2 b) {
  F2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}
__device__ __forceinline__ F2 f2_fma_rn(F2 a, F2 b, F2 c) {
  F2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return d;
}
__device__ __forceinline__ F2 f2_add_rz(F2 a, F2 b) {
  F2 d;
  asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d.v) : "l"(a.v), "l"(b.v));
  return d;
}
__device__ __forceinline__ F2 f2_fma_rz(F2 a, F2 b, F2 c) {
  F2 d;
  asm("fma.rz.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return d;
}

// fixed_weight_parts on two logits at once: the same operations in the same
// order, two lanes per instruction (the clamp and the integer steps per lane).
__device__ __forceinline__ void fixed_weight_parts2(F2 l, F2 Mp, F2 cp, uint32_t& A, uint32_t& Bs) {
  F2 x = f2_mul_rn(f2_sub_rn(l, Mp), cp);
  x = f2(fmaxf(x.lo(), -60.0f), fmaxf(x.hi(), -60.0f));
  const F2 K = f2(12582912.0f, 12582912.0f);
  const F2 t = f2_add_rn(x, K);
  const F2 f = f2_sub_rn(x, f2_sub_rn(t, K));
  F2 p = f2(1.525273365e-05f, 1.525273365e-05f);
  p = f2_fma_rn(p, f, f2(1.540352969e-04f, 1.540352969e-04f));
  p = f2_fma_rn(p, f, f2(1.333355787e-03f, 1.333355787e-03f));
  p = f2_fma_rn(p, f, f2(9.618128650e-03f, 9.618128650e-03f));
  p = f2_fma_rn(p, f, f2(5.550410971e-02f, 5.550410971e-02f));
  p = f2_fma_rn(p, f, f2(2.402265072e-01f, 2.402265072e-01f));
  p = f2_fma_rn(p, f, f2(6.931471825e-01f, 6.931471825e-01f));
  p = f2_fma_rn(p, f, f2(1.0f, 1.0f));
  const F2 sc = f2(__uint_as_float((__float_as_uint(t.lo()) << 23) + (144u << 23)),
                   __uint_as_float((__float_as_uint(t.hi()) << 23) + (144u << 23)));
  const F2 yp = f2_mul_rn(p, sc);
  const F2 two23 = f2(8388608.0f, 8388608.0f);
  const F2 t1 = f2_add_rz(yp, two23);
  const F2 fr = f2_sub_rn(yp, f2_sub_rn(t1, two23));
  const F2 t2 = f2_fma_rz(fr, two23, two23);
  A += __float_as_uint(t1.lo()) + __float_as_uint(t1.hi());
  Bs += __float_as_uint(t2.lo()) + __float_as_uint(t2.hi());
}

// The weights of the 8 logits of a 16-byte vector, summed.  Each sum of 8 a's
// (< 2^21) and 8 b's (< 2^26) is taken modulo 2^32 with the 8 biases removed
// at the end, which is exact because the true sums fit.
__device__ __forceinline__ uint64_t vec_weight(const uint4& v, const WeightParams& wp) {
  uint32_t A = 0u, Bs = 0u;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const F2 Mp = f2(wp.M, wp.M), cp = f2(wp.c, wp.c);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    fixed_weight_parts2({static_cast<uint64_t>(w[k] & 0xFFFF0000u) << 32 | static_cast<uint64_t>(w[k] << 16)}, Mp,
                        cp, A, Bs);
  A -= 8u * 0x4B000000u;
  Bs -= 8u * 0x4B000000u;
  return (static_cast<uint64_t>(A) << 23) + Bs;
}

// One logit's weight (bf16 bits).
__device__ __forceinline__ uint64_t fixed_weight1(uint32_t bits, const WeightParams& wp) {
  uint32_t A = 0u, Bs = 0u;
  fixed_weight_parts(bf16_bits_to_float(bits & 0xFFFFu), wp, A, Bs);
  return (static_cast<uint64_t>(A - 0x4B000000u) << 23) + (Bs - 0x4B000000u);
}

// The float of a bf16 order image (inverse of bf16_order); NaN for 0, the image
// of a row with no non-NaN logit.
__device__ __forceinline__ float order_to_float(uint32_t o) {
  if (o == 0u) return __uint_as_float(0x7FC00000u);
  return bf16_bits_to_float((o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu));
}


__device__ __forceinline__ uint32_t warp_max_u32(uint32_t k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = max(k, __shfl_xor_sync(0xFFFFFFFFu, k, o));
  return k;
}


__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
  return x;
}

// Inclusive prefix sum over the warp's lanes (every lane calls).
__device__ __forceinline__ uint64_t warp_scan_u64(uint64_t x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
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
  int32_t* first_reject;   // = accept_len at the end
  int32_t* out_tok;
  unsigned long long* rowval;   // T = 0: the row's largest key; T > 0: Z
  uint32_t* rowmax;             // T > 0: order image of the row's largest logit
  uint32_t* decided;            // T > 0: 1 once the row's accept test is done
  unsigned long long* slices;   // T > 0: [rows, 8] slice weight sums
  unsigned long long* runs;     // T > 0: [rows, 8, 16] warp-run weight sums
  unsigned* bar;           // T = 0: [0] the count of CTAs done
  uint32_t* err;
};

// ===========================================================================
// T = 0
// ===========================================================================
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

__global__ void verify_init_kernel(int32_t* first_reject, unsigned long long* rowval, uint32_t* decided,
                                   unsigned* bar, int64_t B, int64_t L, int sampled) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = B * (L + 1);
  if (i < B) first_reject[i] = static_cast<int32_t>(L);
  if (!sampled && i < rows) rowval[i] = 0ull;
  if (sampled && i < rows) decided[i] = 0u;
  if (i < 4) bar[i] = 0u;   // the T = 0 count (and three spare words)
}

__global__ void __launch_bounds__(kVThreads, kVCtasPerSm) verify_greedy_kernel(const VerifyArgs a) {
  __shared__ int last_cta;
  pdl_wait();   // no-op: a cooperative launch starts after the init kernel completes
  pdl_launch_dependents();   // lets the next kernel prepare
  const int64_t B = a.B, L = a.L, V = a.V;
  const int nch = verify_chunks(V);
  const int64_t cs = verify_chunk_ids(V);
  volatile int32_t* fr = a.first_reject;
  const int lane = threadIdx.x & 31;
  {
    // item = (t * nch + ch) * B + b: position-major, the sequence fastest, so a
    // sequence's chunks fall on warps of different CTAs (and SMs) and the work
    // of the sequences still alive stays spread over the GPU.  Items are stepped
    // by carry-adds of precomputed (t, ch, b) offsets, so the loop divides nothing.
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
      if (lane == 0 && t < L) {
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
      const uint64_t key = warp_chunk_argmax<kVUnroll>(v, rv, v0, v1, row, lane);
      if (lane == 0) {
        if (key) atomicMax(a.rowval + ri, static_cast<unsigned long long>(key));
        // a key above the draft token's rejects the row (an id outside [0, V)
        // is never the arg-max)
        if (t < L && (dt < 0 || dt >= V || key > id_key(dbits, static_cast<uint32_t>(dt))))
          atomicMin(a.first_reject + b, static_cast<int32_t>(t));
      }
      cur = item_add(cur, stride, nch, Bi);
    }
  }
  // Every thread's atomics are ordered before its CTA's count by fences; the
  // CTA that brings the count to gridDim.x has seen all of them.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_cta = atomicAdd(a.bar, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!last_cta) return;
  __threadfence();
  // n = first_reject[b]: the accepted prefix, row n's token, then -1
  for (int64_t b = threadIdx.x; b < B; b += blockDim.x) {
    const int32_t n = fr[b];
    for (int64_t t = 0; t <= L; ++t) {
      if (t < n) {
        a.out_tok[b * (L + 1) + t] = a.draft_tok[b * L + t];
      } else if (t == n) {
        // row n's largest key (an all-NaN row's is its lowest id's, so 0 only if empty)
        const unsigned long long key = __ldcg(a.rowval + b * (L + 1) + t);
        a.out_tok[b * (L + 1) + t] = key ? static_cast<int32_t>(~static_cast<uint32_t>(key)) : 0;
      } else {
        a.out_tok[b * (L + 1) + t] = -1;
      }
    }
    a.first_reject[b] = n + 1;
  }
}

// ===========================================================================
// T > 0: the rows
// ===========================================================================
struct RowSmem {
  uint64_t bar[2];              // one mbarrier per buffer
  int64_t next_row;             // written by rank 0 into every rank
  float M;                      // the row's maximum (this CTA's copy)
  uint32_t max_part;            // this CTA's slice maximum (order image)
  uint64_t sum_part[kRowCluster];   // rank 0: the slices' weight sums
  uint32_t red32[kRowWarps];
  uint64_t red64[kRowWarps];
};

__device__ __forceinline__ uint32_t block_max_u32(uint32_t x, uint32_t* red) {
  x = warp_max_u32(x);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  uint32_t m = red[0];
#pragma unroll
  for (int w = 1; w < kRowWarps; ++w) m = max(m, red[w]);
  return m;
}

__device__ __forceinline__ uint64_t block_sum_u64(uint64_t x, uint64_t* red) {
  x = warp_sum_u64(x);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  uint64_t t = 0ull;
#pragma unroll
  for (int w = 0; w < kRowWarps; ++w) t += red[w];
  return t;
}

// The largest order image among the bf16 values of smem[0, n) (n % 8 == 0 for
// the vector part; the rest element by element).
__device__ __forceinline__ uint32_t smem_max(const uint16_t* buf, int n) {
  const int nv = n >> 3;
  const uint4* v = reinterpret_cast<const uint4*>(buf);
  uint32_t m = 0u;
  for (int i = threadIdx.x; i < nv; i += kRowThreads) m = max(m, bf16_order(vec_max_bits(v[i])));
  for (int e = nv * 8 + threadIdx.x; e < n; e += kRowThreads) m = max(m, bf16_order(buf[e]));
  return m;
}

// A slice of len ids is split into kRowWarps contiguous warp runs of nvw =
// ceil(len / 8 / kRowWarps) 16-byte vectors each (fewer at the end); the last
// run also takes the slice's last ids that do not fill a vector.  The draw
// reads the runs' sums, so both kernels use this split.
__host__ __device__ __forceinline__ int64_t warp_run_vecs(int64_t len) {
  return ((len >> 3) + kRowWarps - 1) / kRowWarps;
}

// This lane's part of warp w's run inside the piece of slice offsets
// [q0, q1) held in buf: vectors strided by 32 lanes, and (last warp) the ids
// after the slice's last full vector.
__device__ __forceinline__ uint64_t smem_run_sum(const uint16_t* buf, int64_t q0, int64_t q1, int64_t len,
                                                 const WeightParams& wp, int w, int lane) {
  const int64_t nvs = len >> 3, nvw = warp_run_vecs(len);
  const int64_t r0 = imin64(w * nvw, nvs), r1 = imin64(r0 + nvw, nvs);
  const int64_t a = imin64(imax64(r0, q0 >> 3), q1 >> 3), b = imin64(imax64(r1, q0 >> 3), q1 >> 3);
  const uint4* v = reinterpret_cast<const uint4*>(buf) - (q0 >> 3);
  uint64_t acc = 0ull;
#pragma unroll 1
  for (int64_t i = a + lane; i < b; i += 32) acc += vec_weight(v[i], wp);
  if (w == kRowWarps - 1)
    for (int64_t e = imax64(nvs * 8, q0) + lane; e < q1; e += 32) acc += fixed_weight1(buf[e - q0], wp);
  return acc;
}

// A cluster barrier whose release side is paid only by the threads that wrote
// something another CTA reads after it: they fence at cluster scope, every
// thread then arrives relaxed and waits with acquire.  (A full release arrive
// from every thread costs several times more per row.)  Whole-CTA call.
__device__ __forceinline__ void cluster_sync_writers(bool wrote) {
  if (wrote) asm volatile("fence.acq_rel.cluster;" ::: "memory");
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// Row r = t B + b (position-major); whether it still matters.
__device__ __forceinline__ bool row_live(int64_t r, int64_t B, const volatile int32_t* fr) {
  const int64_t t = r / B, b = r - t * B;
  return t <= fr[b];
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Warp 0 of rank 0: the first row among from, from + step, ... (R if none)
// that is live and whose predecessor (the same sequence one position earlier)
// has been decided, so that no row is summed on speculation.  Dead rows are
// checked 32 per round trip.  A live row whose predecessor is undecided is
// waited for (bounded): that predecessor belongs to a cluster that holds no
// undecided row while it waits, so every such chain ends at position 0, which
// never waits.  A wait that passes the limit raises DFLASH2_DEVERR_TIMEOUT and
// ends the cluster's rows (R).  Every lane of the warp calls and gets the answer.
__device__ int64_t next_ready_row(int64_t from, int64_t step, int64_t R, int64_t B, const volatile int32_t* fr,
                                  const uint32_t* decided, uint32_t* err, int lane) {
  for (int64_t base = from; base < R;) {
    const int64_t r0 = base + lane * step;
    const unsigned live = __ballot_sync(0xFFFFFFFFu, r0 < R && row_live(r0, B, fr));
    if (!live) {
      base += 32 * step;
      continue;
    }
    const int64_t r = base + static_cast<int64_t>(__ffs(live) - 1) * step;
    if (r < B) return r;   // position 0: no predecessor
    int ok = 0;
    if (lane == 0) {
      const uint64_t start = global_timer_ns();
      for (;;) {
        if (ld_acquire_u32(decided + (r - B))) {
          ok = row_live(r, B, fr) ? 1 : 0;
          break;
        }
        if (!row_live(r, B, fr)) break;
        if (global_timer_ns() - start > kWaitLimitNs) {
          raise_error(err, DFLASH2_DEVERR_TIMEOUT);
          ok = -1;
          break;
        }
        __nanosleep(100);
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (ok > 0) return r;
    if (ok < 0) return R;
    base = r + step;
  }
  return R;
}

// The piece stream of one CTA: pieces of up to kPieceIds ids of its slice,
// each brought into one of two shared-memory buffers by a bulk copy of its
// 16-byte-aligned part (thread 0) completing on the buffer's mbarrier; the
// piece's last ids (fewer than 8, only at the end of the row) are read
// directly after the wait.  A buffer's phase flips at every completed wait.
struct PieceStream {
  uint16_t* buf[2];
  uint64_t* bar;
  uint32_t phase[2];
  int failed;                   // a wait gave up: no further copies are issued
  uint64_t policy;

  // request piece [p0, p1) of `row` into buffer k (thread 0; the buffer's
  // previous contents must no longer be read)
  __device__ void request(int k, const uint16_t* row, int64_t p0, int64_t p1) {
    if (threadIdx.x != 0) return;
    const uint32_t bytes = static_cast<uint32_t>(((p1 - p0) >> 3) << 4);
    if (bytes == 0u || failed) {
      mbar_arrive(&bar[k]);
    } else {
      // order the CTA's earlier generic accesses of the buffer (seen by this
      // thread through the preceding barrier) before the copy's writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&bar[k], bytes);
      bulk_g2s(buf[k], row + p0, bytes, &bar[k], policy);
    }
  }
  // wait for buffer k, then fill the piece's unaligned tail; whole-CTA call
  __device__ void wait(int k, const uint16_t* row, int64_t p0, int64_t p1, uint32_t* err) {
    if (!mbar_wait_bounded(&bar[k], phase[k], err)) {
      // leave no copy in flight into this CTA's shared memory
      mbar_wait_bounded(&bar[k], phase[k], err);
      failed = 1;
    }
    phase[k] ^= 1u;
    const int64_t full = (p1 - p0) & ~int64_t(7);
    if (threadIdx.x < p1 - p0 - full) buf[k][full + threadIdx.x] = row[p0 + full + threadIdx.x];
    __syncthreads();
  }
};

__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) verify_rows_kernel(const VerifyArgs a) {
  extern __shared__ __align__(128) uint8_t dyn_smem[];
  __shared__ RowSmem s;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t B = a.B, L = a.L, V = a.V;
  const int64_t R = B * (L + 1);
  const float c = __fdiv_rn(kLog2e, a.temperature);
  volatile int32_t* fr = a.first_reject;
  const int64_t ncl = gridDim.x / kRowCluster;
  const int64_t cl = blockIdx.x / kRowCluster;
  // this CTA's slice of every row, and its pieces
  const int64_t sl = verify_slice_ids(V);
  const int64_t s0 = imin64(static_cast<int64_t>(rank) * sl, V), s1 = imin64(s0 + sl, V);
  const int np = static_cast<int>((s1 - s0 + kPieceIds - 1) / kPieceIds);
  PieceStream ps;
  ps.buf[0] = reinterpret_cast<uint16_t*>(align_smem<128>(dyn_smem));
  ps.buf[1] = ps.buf[0] + (kRowBuffers - 1) * kPieceIds;
  ps.bar = s.bar;
  ps.phase[0] = ps.phase[1] = 0u;
  ps.failed = 0;
  ps.policy = np <= 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
  auto piece = [&](int k, int64_t* p0, int64_t* p1) {
    *p0 = s0 + static_cast<int64_t>(k) * kPieceIds;
    *p1 = imin64(*p0 + kPieceIds, s1);
  };
  auto row_ptr = [&](int64_t r) {
    const int64_t t = r / B, b = r - t * B;
    return a.target + (b * (L + 1) + t) * a.ld;
  };
  if (threadIdx.x == 0) {
    mbar_init(&s.bar[0], 1);
    mbar_init(&s.bar[1], 1);
    fence_mbar_init();
  }
  pdl_wait();
  cluster.sync();   // every CTA of the cluster runs before any shared memory is touched remotely
  // the cluster's first row (rank 0 picks for the cluster)
  if (rank == 0 && threadIdx.x < 32) {
    const int64_t r = next_ready_row(cl, ncl, R, B, fr, a.decided, a.err, threadIdx.x);
    if (threadIdx.x < kRowCluster) *cluster.map_shared_rank(&s.next_row, threadIdx.x) = r;
  }
  cluster.sync();
  int64_t r = s.next_row;
  int x = 0;   // the buffer holding (or about to hold) piece 0 of row r
  if (r < R && np == 1) {
    int64_t p0, p1;
    piece(0, &p0, &p1);
    ps.request(0, row_ptr(r), p0, p1);
  }
  while (r < R) {
    const int64_t t = r / B, b = r - t * B;
    const uint16_t* row = row_ptr(r);
    // rank 0 holds the accept test's inputs while the slices stream in
    int32_t xtok = 0, slot = 0;
    uint32_t lx = 0u;
    float q = 0.0f;
    if (rank == 0 && threadIdx.x == 0 && t < L) {
      xtok = a.draft_tok[b * L + t];
      slot = a.draft_slot[b * L + t];
      if (slot < 0 || slot >= kTopK) {
        raise_error(a.err, DFLASH2_DEVERR_BAD_SLOT);
        slot = slot < 0 ? 0 : kTopK - 1;
      }
      q = a.draft_q[(b * L + t) * kTopK + slot];
      if (xtok >= 0 && xtok < V) lx = row[xtok];
      else raise_error(a.err, DFLASH2_DEVERR_BAD_TOKEN);
    }
    // ---- the slice's maximum
    uint32_t m = 0u;
    if (np == 1) {
      int64_t p0, p1;
      piece(0, &p0, &p1);
      ps.wait(x, row, p0, p1, a.err);
      m = smem_max(ps.buf[x], static_cast<int>(p1 - p0));
    } else if (np > 1) {
      for (int k = 0; k < np; ++k) {
        const int kb = k % kRowBuffers;
        int64_t p0, p1;
        if (k == 0 || kRowBuffers == 1) {
          piece(k, &p0, &p1);
          ps.request(kb, row, p0, p1);
        }
        if (kRowBuffers == 2 && k + 1 < np) {
          int64_t q0, q1;
          piece(k + 1, &q0, &q1);
          ps.request((k + 1) % kRowBuffers, row, q0, q1);
        }
        piece(k, &p0, &p1);
        ps.wait(kb, row, p0, p1, a.err);
        m = max(m, smem_max(ps.buf[kb], static_cast<int>(p1 - p0)));
        __syncthreads();   // the buffer is read before it is requested again
      }
    }
    m = block_max_u32(m, s.red32);
    if (threadIdx.x == 0) s.max_part = m;
    cluster_sync_writers(threadIdx.x == 0);   // #1: the slice maxima are in
    if (threadIdx.x == 0) {
      uint32_t mo = 0u;
      for (int k = 0; k < kRowCluster; ++k) mo = max(mo, *cluster.map_shared_rank(&s.max_part, k));
      s.M = order_to_float(mo);
      if (rank == 0) a.rowmax[r] = mo;
    }
    __syncthreads();
    const WeightParams wp(s.M, c);
    // ---- the slice's exact weight sum, by warp runs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t sum = 0ull;
    if (np == 1) {
      sum = smem_run_sum(ps.buf[x], 0, s1 - s0, s1 - s0, wp, warp, lane);
    } else if (np > 1) {
      for (int k = 0; k < np; ++k) {
        const int kb = k % kRowBuffers;
        int64_t p0, p1;
        if (k == 0 || kRowBuffers == 1) {
          piece(k, &p0, &p1);
          ps.request(kb, row, p0, p1);
        }
        if (kRowBuffers == 2 && k + 1 < np) {
          int64_t q0, q1;
          piece(k + 1, &q0, &q1);
          ps.request((k + 1) % kRowBuffers, row, q0, q1);
        }
        piece(k, &p0, &p1);
        ps.wait(kb, row, p0, p1, a.err);
        sum += smem_run_sum(ps.buf[kb], p0 - s0, p1 - s0, s1 - s0, wp, warp, lane);
        __syncthreads();
      }
    }
    sum = warp_sum_u64(sum);
    if (lane == 0) a.runs[(r * kRowCluster + rank) * kRowWarps + warp] = sum;
    sum = block_sum_u64(lane == 0 ? sum : 0ull, s.red64);

    if (threadIdx.x == 0) {
      a.slices[r * kRowCluster + rank] = sum;
      *cluster.map_shared_rank(&s.sum_part[rank], 0) = sum;
    }
    cluster_sync_writers(threadIdx.x == 0);   // #2: the slice sums are in rank 0
    if (rank == 0 && threadIdx.x < 32) {
      if (threadIdx.x == 0) {
        uint64_t Z = 0ull;
        for (int k = 0; k < kRowCluster; ++k) Z += s.sum_part[k];
        a.rowval[r] = Z;
        if (t < L && t <= fr[b]) {
          const uint64_t wx = (xtok >= 0 && xtok < V) ? fixed_weight1(lx, wp) : 0ull;
          const double u1 = philox_uniform24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(t), 1, a.offset);
          if (!(__dmul_rn(__dmul_rn(u1, static_cast<double>(q)), __ull2double_rn(Z)) < __ull2double_rn(wx)))
            atomicMin(a.first_reject + b, static_cast<int32_t>(t));
        }
        __threadfence();
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.decided + r), "r"(1u) : "memory");
      }
      __syncwarp();
      // then the cluster's next row, for every rank
      const int64_t nr = next_ready_row(r + ncl, ncl, R, B, fr, a.decided, a.err, threadIdx.x);
      if (threadIdx.x < kRowCluster) *cluster.map_shared_rank(&s.next_row, threadIdx.x) = nr;
    }
    cluster_sync_writers(rank == 0 && threadIdx.x < kRowCluster);   // #3: the next row is in
    const int64_t nr = s.next_row;
    if (nr < R && np == 1) {
      int64_t p0, p1;
      piece(0, &p0, &p1);
      ps.request(x, row_ptr(nr), p0, p1);
    }
    r = nr;
  }
  // every requested copy was waited for: none is in flight when the CTA leaves
  pdl_launch_dependents();
}

// ===========================================================================
// T > 0: the draws
// ===========================================================================
struct DrawSmem {
  int pick;
  int nc;                       // candidates that correct the weights (0: the draw uses W)
  int64_t lo, hi;               // the picked warp run's ids
  int32_t token;
  uint64_t target;              // the draw's target inside the picked range
  uint64_t red[kDrawThreads / 32];
  int32_t cand[kTopK];          // the rejected row's candidate ids (clamped)
  uint64_t cand_q[kTopK];       // Q_j = floor(min(q_j, 1) Z)
  uint64_t cand_r[kTopK];       // first slot of an id: its residual weight
  uint64_t cand_d[kTopK];       // first slot of an id: residual - weight (mod 2^64); else 0
  int cand_first[kTopK];
  uint64_t cand_w[kTopK];       // the candidate's own weight W
  uint64_t ss[kRowCluster];                 // the row's slice sums (from the rows kernel)
  uint64_t rs[kRowCluster * kRowWarpsC];    // its warp-run sums
  uint64_t runs[kDrawThreads];  // mass of each thread's run of vectors
  uint4 keep[kDrawKeep][kDrawThreads];      // each thread's run vectors, when they fit
};

// Inverse CDF over n <= 256 integer masses mass[0..n) in order (warp 0, 8 per
// lane): the smallest i whose inclusive prefix exceeds tgt (below the total),
// written to s.pick with tgt minus the exclusive prefix to s.target.
__device__ void warp_pick_mass(DrawSmem& s, const uint64_t* mass, int n, uint64_t tgt, int lane) {
  uint64_t loc[8], acc = 0ull;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = lane * 8 + k;
    acc += i < n ? mass[i] : 0ull;
    loc[k] = acc;
  }
  const uint64_t excl = warp_scan_u64(acc, lane) - acc;
  int hit = -1;
#pragma unroll
  for (int k = 7; k >= 0; --k)
    if (tgt < excl + loc[k]) hit = k;
  const unsigned any = __ballot_sync(0xFFFFFFFFu, hit >= 0);
  // exact sums keep tgt below the total, so some lane hits; the fallback is the last entry
  const int src = any ? __ffs(any) - 1 : 31;
  if (lane == src) {
    const int k = hit >= 0 ? hit : 7;
    s.pick = lane * 8 + k;
    s.target = tgt - (excl + (k > 0 ? loc[k - 1] : 0ull));
  }
}

// The row's arg-max id in top-k order (NaN below -inf, lowest id on ties): the
// token of a row with no positive weight.  Whole-CTA call.
__device__ int32_t row_argmax(DrawSmem& s, const uint16_t* row, int64_t V) {
  uint64_t key = 0ull;
  for (int64_t v = threadIdx.x; v < V; v += kDrawThreads) key = kmax(key, id_key(row[v], static_cast<uint32_t>(v)));
  key = warp_max_u64(key);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.red[threadIdx.x >> 5] = key;
  __syncthreads();
  uint64_t k = 0ull;
#pragma unroll
  for (int w = 0; w < kDrawThreads / 32; ++w) k = kmax(k, s.red[w]);
  return static_cast<int32_t>(~static_cast<uint32_t>(k));
}

// The residual correction of ids [lo, hi): the sum of the first-slot deltas of
// candidates in the range (mod 2^64).
__device__ __forceinline__ uint64_t cand_delta(const DrawSmem& s, int nc, int64_t lo, int64_t hi) {
  uint64_t d = 0ull;
  for (int j = 0; j < nc; ++j)
    if (s.cand_first[j] && s.cand[j] >= lo && s.cand[j] < hi) d += s.cand_d[j];
  return d;
}

// Token of row n of sequence b: from the residual after a rejection (n < L),
// from W for the bonus row.  Whole-CTA call.
__device__ int32_t draw_row(DrawSmem& s, const VerifyArgs& a, const uint16_t* row, const unsigned long long* ssum,
                            const unsigned long long* rsum, float M, float c, uint64_t Z, int64_t b, int64_t n) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t V = a.V, L = a.L;
  if (Z == 0ull) return row_argmax(s, row, V);   // no finite logit
  const WeightParams wp(M, c);
  const int nc0 = n < L ? kTopK : 0;
  // each candidate slot takes Q_j off its id; the first slot of an id carries
  // the id's residual and its change of mass
  // (the slice and warp-run sums load meanwhile)
  if (tid < kTopK) {
    int32_t id = 0;
    uint64_t Q = 0ull, w = 0ull;
    if (tid < nc0) {
      id = clamp_token(a.cand_idx[(b * L + n) * kTopK + tid], V, a.err);
      const float qj = a.draft_q[(b * L + n) * kTopK + tid];
      const double qc = qj > 0.0f ? fmin(static_cast<double>(qj), 1.0) : 0.0;
      Q = __double2ull_rz(__dmul_rn(qc, __ull2double_rn(Z)));
      w = fixed_weight1(row[id], wp);
    }
    s.cand[tid] = id;
    s.cand_q[tid] = Q;
    s.cand_w[tid] = w;
  } else if (tid >= 32 && tid < 32 + kRowCluster * kRowWarpsC) {
    s.rs[tid - 32] = __ldcg(rsum + (tid - 32));
  } else if (tid >= 128 && tid < 128 + kRowCluster) {
    s.ss[tid - 128] = __ldcg(ssum + (tid - 128));
  }
  __syncthreads();
  if (tid < kTopK) {
    int first = tid < nc0;
    uint64_t r = 0ull, dlt = 0ull;
    if (tid < nc0) {
      uint64_t qs = 0ull;
      for (int i = 0; i < nc0; ++i)
        if (s.cand[i] == s.cand[tid]) {
          qs += s.cand_q[i];
          if (i < tid) first = 0;
        }
      const uint64_t w = s.cand_w[tid];
      r = w > qs ? w - qs : 0ull;
      dlt = r - w;
    }
    s.cand_first[tid] = first;
    s.cand_r[tid] = r;
    s.cand_d[tid] = first ? dlt : 0ull;
  }
  __syncthreads();
  // the slices' residual masses and their total (warp 0, lane k: slice k);
  // without residual mass (or for the bonus row) the draw uses W itself
  const int64_t sl = verify_slice_ids(V);
  if (tid < 32) {
    int nc = nc0;
    const int k = lane & (kRowCluster - 1);
    const int64_t lo = imin64(k * sl, V), hi = imin64(lo + sl, V);
    const uint64_t base = s.ss[k];
    uint64_t m = base + cand_delta(s, nc, lo, hi);
    uint64_t total = warp_sum_u64(lane < kRowCluster ? m : 0ull);
    if (nc > 0 && total == 0ull) nc = 0;
    if (nc == 0) {
      m = base;
      total = Z;
    }
    const uint64_t U2 = philox_bits24(a.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(n), 2, a.offset);
    // floor(U2 total / 2^24), exactly: U2 < 2^24
    const uint64_t tgt = (__umul64hi(U2, total) << 40) | ((U2 * total) >> 24);
    // the slice: the first whose inclusive prefix exceeds the target
    const uint64_t incl = warp_scan_u64(lane < kRowCluster ? m : 0ull, lane);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < kRowCluster && tgt < incl);
    const int ks = hit ? __ffs(hit) - 1 : kRowCluster - 1;
    uint64_t t2 = tgt - (__shfl_sync(0xFFFFFFFFu, incl, ks) - __shfl_sync(0xFFFFFFFFu, m, ks));
    // the warp run inside it (lane w: run w), from the rows kernel's run sums
    const int64_t d0 = imin64(ks * sl, V), d1 = imin64(d0 + sl, V);
    const int64_t nvs = (d1 - d0) >> 3, nvw = warp_run_vecs(d1 - d0);
    const int w = lane & (kRowWarps - 1);
    const int64_t r0 = d0 + imin64(w * nvw, nvs) * 8;
    const int64_t r1 = w == kRowWarps - 1 ? d1 : d0 + imin64(imin64(w * nvw, nvs) + nvw, nvs) * 8;
    const uint64_t rm = s.rs[ks * kRowWarps + w] + cand_delta(s, nc, r0, r1);
    const uint64_t rincl = warp_scan_u64(lane < kRowWarps ? rm : 0ull, lane);
    const unsigned rhit = __ballot_sync(0xFFFFFFFFu, lane < kRowWarps && t2 < rincl);
    const int rw = rhit ? __ffs(rhit) - 1 : kRowWarps - 1;
    t2 -= __shfl_sync(0xFFFFFFFFu, rincl, rw) - __shfl_sync(0xFFFFFFFFu, rm, rw);
    if (lane == 0) {
      s.nc = nc;
      s.target = t2;
      s.lo = d0 + imin64(rw * nvw, nvs) * 8;
      s.hi = rw == kRowWarps - 1 ? d1 : d0 + imin64(imin64(rw * nvw, nvs) + nvw, nvs) * 8;
    }
  }
  __syncthreads();
  const int nc = s.nc;
  const int64_t lo = s.lo, hi = s.hi;
  // thread runs of contiguous vectors of the warp run (the last thread's run
  // also takes the ids that do not fill a vector)
  const int64_t nv = (hi - lo) >> 3;
  const int64_t per = (nv + kDrawThreads - 1) / kDrawThreads;
  auto run_range = [&](int th, int64_t* rlo, int64_t* rhi) {
    const int64_t i0 = imin64(th * per, nv), i1 = imin64(i0 + per, nv);
    *rlo = lo + i0 * 8;
    *rhi = th == kDrawThreads - 1 ? hi : lo + i1 * 8;
  };
  {
    int64_t tlo, thi;
    run_range(tid, &tlo, &thi);
    uint64_t m = cand_delta(s, nc, tlo, thi);
    const uint4* rv = reinterpret_cast<const uint4*>(row + lo);
    const int64_t i0 = (tlo - lo) >> 3, i1 = imin64((thi - lo) >> 3, nv);
    for (int64_t i = i0; i < i1; i += 8) {
      uint4 vv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) vv[k] = i + k < i1 ? ldg_stream(rv + i + k) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (i + k < i1) {
          m += vec_weight(vv[k], wp);
          if (per <= kDrawKeep && k < kDrawKeep) s.keep[k][tid] = vv[k];
        }
    }
    for (int64_t e = lo + nv * 8; tid == kDrawThreads - 1 && e < hi; ++e) m += fixed_weight1(row[e], wp);
    s.runs[tid] = m;
  }
  const uint64_t rtgt = s.target;
  __syncthreads();
  if (tid < 32) {
    warp_pick_mass(s, s.runs, kDrawThreads, rtgt, lane);
    __syncwarp();
    const int th = s.pick;
    uint64_t rt = s.target;
    int64_t tlo, thi;
    run_range(th, &tlo, &thi);
    // the thread run's vectors, 32 at a time (lane j: vector j of the group),
    // then the picked vector's ids (lane k: id k, a candidate at its residual)
    int64_t vlo = tlo;
    for (;;) {
      const int64_t v = vlo + static_cast<int64_t>(lane) * 8;
      uint64_t mv = 0ull;
      if (v < thi) {
        const int64_t ve = imin64(v + 8, thi);
        if (ve - v == 8) {
          // the picked thread's own vectors stayed in shared memory when they fit
          const int64_t kv = (v - tlo) >> 3;
          mv = vec_weight(per <= kDrawKeep ? s.keep[kv][th] : ldg_stream(reinterpret_cast<const uint4*>(row + v)), wp);
        } else {
          for (int64_t e = v; e < ve; ++e) mv += fixed_weight1(row[e], wp);
        }
        mv += cand_delta(s, nc, v, ve);
      }
      const uint64_t incl = warp_scan_u64(mv, lane);
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, rt < incl);
      const uint64_t group = __shfl_sync(0xFFFFFFFFu, incl, 31);
      if (hit || vlo + 32 * 8 >= thi) {
        // exact sums put rt inside this run; the fallback (not reached) is the run's last vector
        const int vj = hit ? __ffs(hit) - 1 : static_cast<int>(imin64((thi - vlo - 1) >> 3, 31));
        rt -= __shfl_sync(0xFFFFFFFFu, incl, vj) - __shfl_sync(0xFFFFFFFFu, mv, vj);
        const int64_t id0 = vlo + static_cast<int64_t>(vj) * 8;
        const int64_t id = id0 + lane;
        uint64_t w = 0ull;
        if (lane < 8 && id < thi) {
          w = fixed_weight1(row[id], wp);
          for (int j = 0; j < nc; ++j)
            if (s.cand_first[j] && s.cand[j] == id) w = s.cand_r[j];
        }
        const uint64_t wincl = warp_scan_u64(w, lane);
        const unsigned h2 = __ballot_sync(0xFFFFFFFFu, lane < 8 && id < thi && rt < wincl);
        if (lane == 0) s.token = static_cast<int32_t>(h2 ? id0 + __ffs(h2) - 1 : id0);
        break;
      }
      rt -= group;
      vlo += 32 * 8;
    }
  }
  __syncthreads();
  return s.token;
}

__global__ void __launch_bounds__(kDrawThreads) verify_draw_kernel(const VerifyArgs a) {
  __shared__ DrawSmem s;
  pdl_wait();
  pdl_launch_dependents();
  const int64_t B = a.B, L = a.L;
  const float c = __fdiv_rn(kLog2e, a.temperature);
  for (int64_t b = blockIdx.x; b < B; b += gridDim.x) {
    const int64_t n = a.first_reject[b];
    const int64_t r = n * B + b;
    const uint16_t* row = a.target + (b * (L + 1) + n) * a.ld;
    const float M = order_to_float(__ldcg(a.rowmax + r));
    const uint64_t Z = __ldcg(a.rowval + r);
    const int32_t tok = draw_row(s, a, row, a.slices + r * kRowCluster, a.runs + r * kRowCluster * kRowWarps, M, c,
                                 Z, b, n);
    // this sequence's outputs: the accepted prefix, row n's token, then -1
    for (int64_t t = threadIdx.x; t <= L; t += kDrawThreads)
      a.out_tok[b * (L + 1) + t] = t < n ? a.draft_tok[b * L + t] : (t == n ? tok : -1);
    __syncthreads();   // every thread has read first_reject[b]
    if (threadIdx.x == 0) a.first_reject[b] = static_cast<int32_t>(n + 1);
  }
}

int max_greedy_grid(int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_greedy_kernel, kVThreads, 0) != cudaSuccess ||
      per_sm < 1)
    return 0;
  return per_sm * num_sms;
}

size_t rows_smem_bytes() { return static_cast<size_t>(kRowBuffers) * kPieceIds * sizeof(uint16_t) + 128; }

int max_row_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kRowCluster, 1, 1);
  cfg.blockDim = dim3(kRowThreads, 1, 1);
  cfg.dynamicSmemBytes = rows_smem_bytes();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRowCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_rows_kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace

int64_t verify_max_vocab() { return 10485760; }

size_t verify_workspace_bytes(int64_t B, int64_t L, int64_t V) {
  (void)V;
  return ScratchLayout(B * (L + 1)).total;
}

cudaError_t launch_verify(const uint16_t* target, int64_t ld, const int32_t* draft_tok,
                          const int32_t* draft_slot, const float* draft_q, const int32_t* cand_idx,
                          int64_t B, int64_t L, int64_t V, float temperature, uint64_t seed,
                          uint64_t offset, int32_t* accept_len, int32_t* out_tok, void* workspace,
                          uint32_t* err, int num_sms, cudaStream_t stream) {
  const int64_t rows = B * (L + 1);
  const int nch = verify_chunks(V);
  if (rows > 0x7FFFFFFFLL / nch) return cudaErrorInvalidValue;
  const bool sampled = temperature > 0.0f;
  const ScratchLayout lay(rows);
  uint8_t* sc = static_cast<uint8_t*>(workspace);
  unsigned* bar = reinterpret_cast<unsigned*>(sc);
  unsigned long long* rowval = reinterpret_cast<unsigned long long*>(sc + lay.rowval);
  VerifyArgs args{target, ld, draft_tok, draft_slot, draft_q, cand_idx, B, L, V, temperature, seed, offset,
                  accept_len, out_tok, rowval, reinterpret_cast<uint32_t*>(sc + lay.rowmax),
                  reinterpret_cast<uint32_t*>(sc + lay.decided), reinterpret_cast<unsigned long long*>(sc + lay.slices),
                  reinterpret_cast<unsigned long long*>(sc + lay.runs), bar, err};
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_init_kernel, accept_len, rowval,
                                             reinterpret_cast<uint32_t*>(sc + lay.decided), bar, B, L, sampled ? 1 : 0);
    if (e != cudaSuccess) return e;
  }
  // the co-resident grid (T = 0) or cluster count (T > 0), per device
  static std::mutex mu;
  static int grid_cache[kMaxDevices][2] = {};
  int dev = 0;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sampled) {
    const cudaError_t se = set_smem_limit<verify_rows_kernel>(rows_smem_bytes());
    if (se != cudaSuccess) return se;
  }
  int g;
  {
    std::lock_guard<std::mutex> lock(mu);
    int& cached = grid_cache[dev][sampled ? 1 : 0];
    if (cached == 0) cached = sampled ? max_row_clusters() : max_greedy_grid(num_sms);
    g = cached;
  }
  if (g == 0) return cudaErrorInvalidConfiguration;
  if (!sampled) {
    const int64_t ctas = ((L + 1) * B * nch + kVWarps - 1) / kVWarps;   // one warp per item at most
    const int grid = static_cast<int>(ctas < g ? ctas : g);
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(verify_greedy_kernel), grid, kVThreads, kargs, 0,
                                       stream);
  }
  {
    // rows: as many clusters as can be resident, none more than there are rows
    const int64_t ncl = rows < g ? rows : g;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * kRowCluster), 1, 1);
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    cfg.dynamicSmemBytes = rows_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kRowCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_rows_kernel, args);
    if (e != cudaSuccess) return e;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B < 65535 ? B : 65535), 1, 1);
    cfg.blockDim = dim3(kDrawThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_draw_kernel, args);
  }
}

}  // namespace dflash2
