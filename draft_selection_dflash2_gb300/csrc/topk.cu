// topk.cu -- per-position top-16 over bf16 logits ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector": keep the top 16 candidates of the
// drafter's own logits at every block position).
//
// Two forms.  Segments of up to kHistSegMax logits (rows up to 196,608 per
// CTA, longer ones split over a larger cluster first) take the group-maximum
// form below (topk16_hist_kernel); longer segments take the running-threshold
// stream (topk16_kernel):
//   * A row is split into `S` contiguous segments, one per CTA of an S-CTA
//     thread-block cluster (S = 1 when there are enough rows to fill the GPU).
//   * The eight warps of a CTA stream the segment in 512-logit blocks (one
//     16-byte vector per lane), interleaved, with kUnroll independent vector
//     loads per lane in flight (ld.global.nc, no L1 allocation); nothing in the
//     streaming loop synchronises, so memory-level parallelism comes from every
//     warp's own outstanding loads.
//   * Each warp keeps its own running top-16 (one key per lane), threshold and
//     candidate buffer.  A packed bf16x2 max over each lane's 8 logits against
//     max(warp threshold, CTA-wide bound) rejects almost every vector; the rare
//     survivors are turned into exact 64-bit keys (value, -id) out of line and
//     buffered; once a warp holds more than kFoldAt of them it folds them into
//     its top-16 with bitonic merges (survivors appear in most iterations early
//     in a row, so folding on every one would dominate).  After each fold the
//     warp raises the CTA-wide bound (shared memory atomicMax): the CTA's 16th
//     best is at least any warp's 16th best, so the bound is safe for all warps.
//   * At the end the eight warp lists are merged, then the S CTA lists meet in
//     distributed shared memory: CTA rank 0 reads them with ld.shared::cluster,
//     merges and writes the row's output.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace dflash2 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 8;                           // vectors in flight per lane
constexpr int kCtasPerSm = 4;
constexpr int kFoldAt = 32;                          // fold a warp buffer beyond this many
constexpr int kWarpCap = kFoldAt + 32 * 8;           // + one vector from every lane
constexpr int kSegQuantum = 8;                       // segments start on 16-byte boundaries

struct TopkSmem {
  uint64_t cand[kWarps][kWarpCap];
  uint64_t warp_top[kWarps][kTopK];
  uint64_t top[kTopK];
  unsigned long long gthr;   // CTA-wide lower bound on the 16th best key
  int wcount[kWarps];
};

// Max of 8 bf16 values (bf16x2 max; a NaN never wins) as bf16 bits.
__device__ __forceinline__ uint32_t vec_max_bits(uint4 v) {
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&v.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v.y);
  __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&v.z);
  __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&v.w);
  const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
  const __nv_bfloat16 mm = __hmax(__low2bfloat16(m), __high2bfloat16(m));
  return static_cast<uint32_t>(__bfloat16_as_ushort(mm));
}

__device__ __forceinline__ uint32_t lane_elem(const uint4& v, int k) {
  const uint32_t w = (k < 4) ? ((k < 2) ? v.x : v.y) : ((k < 6) ? v.z : v.w);
  return (k & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ uint4 ldg_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The bf16 value whose order-preserving image is `ord` (ord != 0).
__device__ __forceinline__ uint32_t bf16_from_order(uint32_t ord) {
  return (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
}

// Does any of the vector's 8 logits compare >= t2 (both halves hold the
// threshold value)?  NaN never compares; -0 == +0.
__device__ __forceinline__ bool vec_reaches(uint4 v, __nv_bfloat162 t2) {
  const __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&v.x);
  const __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v.y);
  const __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&v.z);
  const __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&v.w);
  return __hge2_mask(__hmax2(__hmax2(a, b), __hmax2(c, d)), t2) != 0u;
}

// Bit k set iff element k of the vector compares >= t2 (NaN never does).
__device__ __forceinline__ uint32_t elem_reach_mask(uint4 v, __nv_bfloat162 t2) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t r = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[q]), t2);
    m |= ((r & 1u) | ((r >> 15) & 2u)) << (2 * q);
  }
  return m;
}

// Per-warp selection state; `top` is distributed (lane i < 16 holds the i-th
// best key, lanes 16..31 hold 0), `thr` is warp-uniform.
struct WarpSel {
  uint64_t top;
  uint64_t thr;
};

// top: a descending top-16 in lanes 0..15 (0 in lanes 16..31); x: a bitonic
// sequence, a descending 16-list in lanes 0..15 and another in reverse
// (ascending) in lanes 16..31.  Returns the top-16 of the three lists: five
// bitonic merge stages sort x (two sorted lists need no full sort), five more
// merge it with top.  Whole warp.
__device__ __forceinline__ uint64_t merge_sorted_pair(uint64_t top, uint64_t x, int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, x, j);
    x = ((lane & j) == 0) ? kmax(x, o) : kmin(x, o);
  }
  const uint64_t xr = __shfl_sync(0xFFFFFFFFu, x, 31 - lane);
  uint64_t c = kmax(top, xr);
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, c, j);
    c = ((lane & j) == 0) ? kmax(c, o) : kmin(c, o);
  }
  return lane < kTopK ? c : 0ull;
}

// Rare path, kept out of line so the streaming loop stays small: appends the
// keys of one lane's vector (first id id0) that beat `thr` to the warp buffer.
__device__ __noinline__ void append_vector(uint64_t* cand, int* wcount, uint4 v, uint32_t id0, uint64_t thr) {
  for (int k = 0; k < 8; ++k) {
    const uint64_t key = make_key(lane_elem(v, k), id0 + k);
    if (key > thr) cand[atomicAdd(wcount, 1)] = key;
  }
}

// Folds the warp's pending candidates into its top-16 and raises the CTA-wide
// bound.  Whole warp.
__device__ __noinline__ void fold_warp(WarpSel& w, uint64_t* cand, int* wcount, unsigned long long* gthr,
                                       int lane) {
  __syncwarp();
  const int n = *reinterpret_cast<volatile int*>(wcount);
  for (int base = 0; base < n; base += 32)
    w.top = warp_merge_top16(w.top, base + lane < n ? cand[base + lane] : 0ull, lane);
  const uint64_t own = __shfl_sync(0xFFFFFFFFu, w.top, kTopK - 1);   // 0 while < 16 candidates
  __syncwarp();
  if (lane == 0) {
    *wcount = 0;
    atomicMax(gthr, static_cast<unsigned long long>(own));
  }
  __syncwarp();
  // the warp threshold never drops below the CTA-wide bound
  const uint64_t g = *reinterpret_cast<volatile unsigned long long*>(gthr);
  w.thr = own > g ? own : g;
}

// The barriers around a row's merge.  A one-CTA cluster needs only the CTA
// barrier; a larger one arrives relaxed, the threads that wrote data another
// CTA reads after the barrier fencing at cluster scope first, and waits with
// acquire.  Whole-CTA call.
__device__ __forceinline__ void merge_sync(unsigned nrank, bool wrote) {
  if (nrank == 1) {
    __syncthreads();
    return;
  }
  if (wrote) asm volatile("fence.acq_rel.cluster;" ::: "memory");
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) topk16_kernel(const uint16_t* __restrict__ logits,
                                                          int64_t V, int64_t ld, int64_t seg_len,
                                                          float* __restrict__ vals,
                                                          int32_t* __restrict__ idx) {
  __shared__ TopkSmem s;
  pdl_wait();
  pdl_launch_dependents();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const unsigned nrank = cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;

  const int64_t seg_begin = static_cast<int64_t>(rank) * seg_len;
  const int64_t seg_end = seg_begin + seg_len < V ? seg_begin + seg_len : V;
  const int64_t n_elems = seg_end > seg_begin ? seg_end - seg_begin : 0;
  const int64_t n_vecs = n_elems >> 3;                 // whole 16-byte vectors
  const uint16_t* seg = logits + row * ld + seg_begin;

  if (tid < kWarps) s.wcount[tid] = 0;
  if (tid == 0) s.gthr = 0ull;
  __syncthreads();

  WarpSel w{0ull, 0ull};
  uint64_t* cand = s.cand[warp];
  int* wcount = &s.wcount[warp];
  // warp `warp` owns blocks warp, warp + 8, ...; lane `lane` owns vector `lane` of each
  const int64_t stride = static_cast<int64_t>(kWarps) * 32;          // vectors between a warp's blocks
  uint4 v[kUnroll];
  int64_t vb = static_cast<int64_t>(warp) * 32;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t vi = vb + u * stride + lane;
    v[u] = vi < n_vecs ? ldg_stream(seg + vi * 8) : make_uint4(0u, 0u, 0u, 0u);
  }
  {
    // Initial CTA-wide bound: the 16th largest of the 256 lane maxima of the
    // first iteration (16 distinct logits reach it); lanes without data give 0.
    uint32_t lm = 0u;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (vb + u * stride + lane < n_vecs) lm = max(lm, bf16_order(vec_max_bits(v[u])));
    const uint64_t sorted = warp_sort_desc(static_cast<uint64_t>(lm) << 48, lane);
    if (lane < kTopK) s.warp_top[warp][lane] = sorted;
    __syncthreads();
    if (warp == 0) {
      uint64_t acc = 0ull;
#pragma unroll
      for (int ww = 0; ww < kWarps; ww += 2) {
        const uint64_t x = (lane < kTopK) ? s.warp_top[ww][lane] : s.warp_top[ww + 1][31 - lane];
        acc = merge_sorted_pair(acc, x, lane);
      }
      if (lane == kTopK - 1) s.gthr = acc;
    }
    __syncthreads();
  }
  for (; vb < n_vecs; vb += stride * kUnroll) {
    // every vector of this iteration exists for every lane (all but a row's last)
    const bool whole = vb + (kUnroll - 1) * stride + 32 <= n_vecs;
    if (vb != static_cast<int64_t>(warp) * 32) {
      const uint4* p = reinterpret_cast<const uint4*>(seg) + (vb + lane);
      if (whole) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ldg_stream(reinterpret_cast<const uint16_t*>(p + u * stride));
      } else {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          v[u] = vb + u * stride + lane < n_vecs ? ldg_stream(reinterpret_cast<const uint16_t*>(p + u * stride))
                                                 : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    const uint64_t g = *reinterpret_cast<volatile unsigned long long*>(&s.gthr);
    if (g > w.thr) w.thr = g;
    const uint32_t thr_ord = static_cast<uint32_t>(w.thr >> 48);
    const uint32_t tb = bf16_from_order(thr_ord);
    const __nv_bfloat162 t2 = __halves2bfloat162(__ushort_as_bfloat16(static_cast<unsigned short>(tb)),
                                                 __ushort_as_bfloat16(static_cast<unsigned short>(tb)));
    uint32_t mask = 0u;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool real = whole || vb + u * stride + lane < n_vecs;
      if (real && (thr_ord == 0u || vec_reaches(v[u], t2))) mask |= 1u << u;
    }
    if (__ballot_sync(0xFFFFFFFFu, mask != 0u) != 0u) {
      if (__reduce_add_sync(0xFFFFFFFFu, static_cast<unsigned>(__popc(mask))) <= 32u) {
        // the usual case: few flagged vectors, and the buffer (at most kFoldAt
        // keys between entries) has room for all their keys; each lane keys only
        // the elements that reach the threshold value
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          if ((mask >> u) & 1u) {
            const uint4 x = v[u];
            const uint32_t id0 = static_cast<uint32_t>(seg_begin + (vb + u * stride + lane) * 8);
            uint32_t em = thr_ord == 0u ? 0xFFu : elem_reach_mask(x, t2);
            while (em) {
              const int k = __ffs(em) - 1;
              em &= em - 1u;
              const uint64_t key = make_key(lane_elem(x, k), id0 + k);
              if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
            }
          }
        }
        __syncwarp();
        if (*reinterpret_cast<volatile int*>(wcount) > kFoldAt) fold_warp(w, cand, wcount, &s.gthr, lane);
        continue;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const bool f = (mask >> u) & 1u;
        if (__ballot_sync(0xFFFFFFFFu, f) == 0u) continue;
        if (f) append_vector(cand, wcount, v[u], static_cast<uint32_t>(seg_begin + (vb + u * stride + lane) * 8), w.thr);
        __syncwarp();
        if (*reinterpret_cast<volatile int*>(wcount) > kFoldAt) fold_warp(w, cand, wcount, &s.gthr, lane);
      }
    }
  }
  // NaN logits need no extra pass: while the threshold is empty every real
  // vector is flagged (and NaN keys, order 0, qualify), and once it is not, a
  // NaN key can never beat it.
  if (warp == 0) {
    const int64_t tail = n_elems - n_vecs * 8;
    if (lane < tail) {
      const int64_t e = n_vecs * 8 + lane;
      const uint64_t key = make_key(seg[e], static_cast<uint32_t>(seg_begin + e));
      if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
    }
  }
  fold_warp(w, cand, wcount, &s.gthr, lane);
  if (lane < kTopK) s.warp_top[warp][lane] = w.top;
  __syncthreads();
  if (warp == 0) {
    uint64_t acc = 0ull;
#pragma unroll
    for (int ww = 0; ww < kWarps; ww += 2) {
      const uint64_t x = (lane < kTopK) ? s.warp_top[ww][lane] : s.warp_top[ww + 1][31 - lane];
      acc = merge_sorted_pair(acc, x, lane);
    }
    if (lane < kTopK) s.top[lane] = acc;
  }

  // Merge the cluster's partial lists in distributed shared memory.
  merge_sync(nrank, warp == 0 && lane < kTopK);
  if (rank == 0 && warp == 0) {
    uint64_t acc = lane < kTopK ? s.top[lane] : 0ull;
    for (unsigned r = 1; r < nrank; r += 2) {
      uint64_t x = 0ull;
      const unsigned src = lane < kTopK ? r : r + 1;
      if (src < nrank) {
        const uint64_t* remote = cluster.map_shared_rank(s.top, src);
        x = remote[lane < kTopK ? lane : 31 - lane];
      }
      acc = merge_sorted_pair(acc, x, lane);
    }
    if (lane < kTopK) {
      vals[row * kTopK + lane] = key_value(acc);
      idx[row * kTopK + lane] = key_id(acc);
    }
  }
  merge_sync(nrank, false);   // rank 0 has read every list before any CTA leaves
}

// ---------------------------------------------------------------------------
// Group-maximum form (segments up to kHistSegMax logits)
// ---------------------------------------------------------------------------
// A thread's 8 vectors of one CTA iteration (64 logits) form a group.  The
// stream keeps for each group (in shared memory) its maximum, where it sits
// (vector and element) with its bits, and the largest of the group's other 63
// logits; a lane's vector is dead once these are updated and its next load is
// issued at once, so the stream runs at close to a plain copy's read rate.
// Then T = the 16th largest of the 256 threads' maxima: those are 16 distinct
// logits >= T, so no logit below T is in the segment's top-16, and every
// logit of the top-16 lies in a group whose maximum reaches T (about 16 of a
// row's 2,400).  A group whose other logits all fall below T holds exactly one
// logit >= T, keyed from the history alone; any other reaching group is read
// again by the thread that streamed it (from L2, as a rule) and its logits
// >= T keyed exactly.  The keys fold into the warp lists; the segment's few
// trailing logits (V % 8) are keyed directly.  Rows of ties (every group
// reaching T) stay exact: their groups are read again, and the folds take any
// number of keys.
constexpr int kHistIters = 12;                                        // CTA iterations a segment may take
constexpr int64_t kHistSegMax = static_cast<int64_t>(kHistIters) * kThreads * kUnroll * 8;

// A group's history entry (0: the thread had no data in that iteration):
//   bits  0..16  bf16 order of the group maximum + 1
//   bits 17..22  where the maximum sits: 8 * vector + element (its first
//                occurrence in the vector that first holds it)
//   bits 23..38  the maximum's own bf16 bits
//   bits 39..54  bf16 order of the largest of the other 63 logits (an upper
//                bound when some are NaN)
//   bit  55      the maximum was located (the group holds a non-NaN logit)
constexpr int kHistMaxBits = 17;

struct HistSmem {
  uint64_t hist[kHistIters][kThreads];
  uint64_t cand[kWarps][kWarpCap];
  uint64_t warp_top[kWarps][kTopK];
  uint64_t top[kTopK];
  unsigned long long gthr;
  uint64_t tkey;                         // the 16th largest thread-maximum key
  int wcount[kWarps];
  int wfold[kWarps];                     // the warp folded its buffer during the re-read
};

__device__ __forceinline__ uint32_t max2_bits(uint32_t a, uint32_t b) {
  const __nv_bfloat162 m = __hmax2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&m);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) topk16_hist_kernel(const uint16_t* __restrict__ logits,
                                                               int64_t V, int64_t ld, int64_t seg_len,
                                                               float* __restrict__ vals,
                                                               int32_t* __restrict__ idx) {
  __shared__ HistSmem s;
  pdl_wait();
  pdl_launch_dependents();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const unsigned nrank = cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;

  const int64_t seg_begin = static_cast<int64_t>(rank) * seg_len;
  const int64_t seg_end = seg_begin + seg_len < V ? seg_begin + seg_len : V;
  const int64_t n_elems = seg_end > seg_begin ? seg_end - seg_begin : 0;
  const int64_t n_vecs = n_elems >> 3;                 // whole 16-byte vectors
  const uint16_t* seg = logits + row * ld + seg_begin;
  constexpr int64_t stride = kThreads;                 // vectors between a thread's vectors in an iteration
  constexpr int64_t per_iter = stride * kUnroll;       // vectors per CTA iteration
  const int iters = static_cast<int>((n_vecs + per_iter - 1) / per_iter);

  if (tid < kWarps) s.wcount[tid] = 0;
  if (tid == 0) s.gthr = 0ull;

  // ---- stream: group histories; a lane reloads each vector as soon as it is reduced
  const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);   // never a maximum
  const __nv_bfloat16 ninf = __ushort_as_bfloat16(static_cast<unsigned short>(0xFF80u));
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t vi = u * stride + tid;
    v[u] = vi < n_vecs ? ldg_stream(seg + vi * 8) : nan4;
  }
  uint32_t lane_max = 0u;   // the largest of this thread's group maxima (order + 1)
  for (int it = 0; it < iters; ++it) {
    const int64_t nb = static_cast<int64_t>(it + 1) * per_iter;
    uint32_t m2 = 0u;
    // the first vector holding the largest vector maximum (NaN taken as -inf
    // here), the vector itself, and the largest maximum of the other vectors
    __nv_bfloat16 best = ninf, rest = ninf;
    int bu = 0;
    uint4 bv = v[0];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w = max2_bits(max2_bits(v[u].x, v[u].y), max2_bits(v[u].z, v[u].w));
      m2 = u == 0 ? w : max2_bits(m2, w);
      const __nv_bfloat162 wb = *reinterpret_cast<const __nv_bfloat162*>(&w);
      const __nv_bfloat16 vm = __hmax(__hmax(__low2bfloat16(wb), __high2bfloat16(wb)), ninf);
      if (u == 0) {
        best = vm;
      } else {
        const bool better = __hgt(vm, best);
        rest = __hmax(rest, better ? best : vm);
        best = better ? vm : best;
        bu = better ? u : bu;
        bv = better ? v[u] : bv;
      }
      const int64_t vi = nb + u * stride + tid;
      v[u] = vi < n_vecs ? ldg_stream(seg + vi * 8) : nan4;
    }
    const __nv_bfloat162 mb = *reinterpret_cast<const __nv_bfloat162*>(&m2);
    const uint32_t gm = __bfloat16_as_ushort(__hmax(__low2bfloat16(mb), __high2bfloat16(mb)));
    const bool has = static_cast<int64_t>(it) * per_iter + tid < n_vecs;
    uint64_t h = has ? bf16_order(gm) + 1u : 0u;
    if (has && bf16_order(gm) != 0u) {
      // the maximum's first element in its vector; the largest of the vector's others
      int k0 = -1;
      __nv_bfloat16 other = ninf;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __nv_bfloat16 e = __ushort_as_bfloat16(static_cast<unsigned short>(lane_elem(bv, k)));
        const bool hit = k0 < 0 && __heq(e, best);
        other = hit ? other : __hmax(other, e);
        k0 = hit ? k : k0;
      }
      if (k0 >= 0) {
        const uint32_t mbits = lane_elem(bv, k0);
        const uint32_t rest_ord = bf16_order(__bfloat16_as_ushort(__hmax(rest, other)));
        h |= (static_cast<uint64_t>(bu * 8 + k0) << kHistMaxBits) | (static_cast<uint64_t>(mbits) << 23) |
             (static_cast<uint64_t>(rest_ord) << 39) | (1ull << 55);
      }
    }
    s.hist[it][tid] = h;
    const uint32_t hm = static_cast<uint32_t>(h) & ((1u << kHistMaxBits) - 1u);
    lane_max = hm > lane_max ? hm : lane_max;
  }

  // ---- T: the 16th largest thread maximum (the maxima of 16 threads are 16
  // distinct logits, so T bounds the segment's 16th best from below)
  {
    const uint64_t key = lane_max ? (static_cast<uint64_t>(lane_max) << 32) | static_cast<uint32_t>(~tid) : 0ull;
    const uint64_t sorted = warp_sort_desc(key, lane);
    if (lane < kTopK) s.warp_top[warp][lane] = sorted;
    __syncthreads();   // also publishes the group entries
    if (warp == 0) {
      uint64_t a2 = 0ull;
#pragma unroll
      for (int ww = 0; ww < kWarps; ww += 2) {
        const uint64_t x = (lane < kTopK) ? s.warp_top[ww][lane] : s.warp_top[ww + 1][31 - lane];
        a2 = merge_sorted_pair(a2, x, lane);
      }
      if (lane == kTopK - 1) s.tkey = a2;
    }
    __syncthreads();
  }
  // fewer than 16 threads with data: every group with data
  const uint32_t T = static_cast<uint32_t>(s.tkey >> 32) > 1u ? static_cast<uint32_t>(s.tkey >> 32) : 1u;
  const uint32_t t_ord = T - 1u;                      // logits of order >= t_ord qualify
  const uint32_t tb = t_ord ? bf16_from_order(t_ord) : 0u;
  const __nv_bfloat162 t2 = __halves2bfloat162(__ushort_as_bfloat16(static_cast<unsigned short>(tb)),
                                               __ushort_as_bfloat16(static_cast<unsigned short>(tb)));

  // ---- the groups that reach T: keyed from the history when they hold one
  // logit >= T, else read again and keyed exactly; each thread takes its own,
  // one group per round, so a warp's first round covers the usual single group
  WarpSel w{0ull, 0ull};
  uint64_t* cand = s.cand[warp];
  int* wcount = &s.wcount[warp];
  auto next_sel = [&](int from) {
    int it = from;
    if (lane_max >= T)
      while (it < iters && (static_cast<uint32_t>(s.hist[it][tid]) & ((1u << kHistMaxBits) - 1u)) < T) ++it;
    else
      it = iters;
    return it;
  };
  int it = next_sel(0);
  while (__ballot_sync(0xFFFFFFFFu, it < iters) != 0u) {
    const bool sel = it < iters;
    const uint64_t hist = sel ? s.hist[it][tid] : 0ull;
    // one logit >= T (t_ord > 0: NaN never reaches it): the located maximum
    const bool lone = sel && t_ord != 0u && ((hist >> 55) & 1ull) && ((hist >> 39) & 0xFFFFull) < t_ord;
    if (lone) {
      const int pos = static_cast<int>((hist >> kHistMaxBits) & 63ull);
      const int64_t vi = static_cast<int64_t>(it) * per_iter + (pos >> 3) * stride + tid;
      const uint64_t key = make_key(static_cast<uint32_t>((hist >> 23) & 0xFFFFull),
                                    static_cast<uint32_t>(seg_begin + vi * 8 + (pos & 7)));
      if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
    }
    __syncwarp();
    if (*reinterpret_cast<volatile int*>(wcount) > kFoldAt) fold_warp(w, cand, wcount, &s.gthr, lane);
    const bool reread = sel && !lone;
    const int64_t b0 = static_cast<int64_t>(reread ? it : 0) * per_iter + tid;
    uint4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) x[u] = reread && b0 + u * stride < n_vecs ? ldg_stream(seg + (b0 + u * stride) * 8) : nan4;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (reread && b0 + u * stride < n_vecs) {
        const uint32_t id0 = static_cast<uint32_t>(seg_begin + (b0 + u * stride) * 8);
        uint32_t em = t_ord == 0u ? 0xFFu : elem_reach_mask(x[u], t2);
        while (em) {
          const int k = __ffs(em) - 1;
          em &= em - 1u;
          const uint64_t key = make_key(lane_elem(x[u], k), id0 + k);
          if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
        }
      }
      __syncwarp();
      if (*reinterpret_cast<volatile int*>(wcount) > kFoldAt) fold_warp(w, cand, wcount, &s.gthr, lane);
    }
    it = sel ? next_sel(it + 1) : iters;
  }
  if (warp == 0) {
    const int64_t tail = n_elems - n_vecs * 8;
    if (lane < tail) {
      const int64_t e = n_vecs * 8 + lane;
      const uint64_t key = make_key(seg[e], static_cast<uint32_t>(seg_begin + e));
      if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
    }
  }
  // Warp 0 merges the lists of the warps that folded (usually none) and then
  // every key still buffered, 32 at a time over all warps' buffers (usually
  // one round), instead of a fold per warp and a merge of eight lists.
  const bool folded = __any_sync(0xFFFFFFFFu, w.top != 0ull);
  if (lane < kTopK) s.warp_top[warp][lane] = w.top;
  if (lane == 0) s.wfold[warp] = folded ? 1 : 0;
  __syncthreads();
  if (warp == 0) {
    uint64_t acc = 0ull;
#pragma unroll
    for (int ww = 0; ww < kWarps; ww += 2) {
      if (!(s.wfold[ww] | s.wfold[ww + 1])) continue;
      const uint64_t x = (lane < kTopK) ? s.warp_top[ww][lane] : s.warp_top[ww + 1][31 - lane];
      acc = merge_sorted_pair(acc, x, lane);
    }
    int cnt[kWarps], total = 0;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      cnt[ww] = s.wcount[ww];
      total += cnt[ww];
    }
    for (int base = 0; base < total; base += 32) {
      int i = base + lane;
      uint64_t key = 0ull;
      if (i < total) {
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
          if (i >= 0 && i < cnt[ww]) key = s.cand[ww][i];
          i -= cnt[ww];
        }
      }
      acc = warp_merge_top16(acc, key, lane);
    }
    if (lane < kTopK) s.top[lane] = acc;
  }
  // the cluster's lists meet in distributed shared memory
  merge_sync(nrank, warp == 0 && lane < kTopK);
  if (rank == 0 && warp == 0) {
    uint64_t acc = lane < kTopK ? s.top[lane] : 0ull;
    for (unsigned r = 1; r < nrank; r += 2) {
      uint64_t x = 0ull;
      const unsigned src = lane < kTopK ? r : r + 1;
      if (src < nrank) {
        const uint64_t* remote = cluster.map_shared_rank(s.top, src);
        x = remote[lane < kTopK ? lane : 31 - lane];
      }
      acc = merge_sorted_pair(acc, x, lane);
    }
    if (lane < kTopK) {
      vals[row * kTopK + lane] = key_value(acc);
      idx[row * kTopK + lane] = key_id(acc);
    }
  }
  merge_sync(nrank, false);   // rank 0 has read every list before any CTA leaves
}
}  // namespace

int topk_cluster_size(int64_t rows, int64_t V, int num_sms) {
  // The CTAs run in waves of kCtasPerSm per SM, each wave as long as its
  // segments.  With rows for at least half the slots, whole rows (a split
  // costs a cluster merge and wave tails, measured slower at 2048 rows);
  // otherwise the split S (segments of at least 8192 logits) that minimises
  // waves x (segment + a fixed cost of about 8192 logits per CTA).
  const int64_t slots = static_cast<int64_t>(kCtasPerSm) * num_sms;
  if (2 * rows >= slots) return 1;
  int best = 1;
  int64_t best_cost = -1;
  for (int S = 1; S <= 16; S <<= 1) {
    if (S > 1 && (V + S - 1) / S < 8192) break;
    const int64_t waves = (rows * S + slots - 1) / slots;
    const int64_t cost = waves * ((V + S - 1) / S + 8192);
    if (best_cost < 0 || cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t launch_topk(const uint16_t* logits, int64_t rows, int64_t V, int64_t ld, float* vals,
                        int32_t* idx, uint32_t* err, int num_sms, cudaStream_t stream) {
  (void)err;
  auto seg_of = [&](int S) {
    const int64_t l = (V + S - 1) / S;
    return (l + kSegQuantum - 1) / kSegQuantum * kSegQuantum;
  };
  // the group-maximum form while a segment fits its shared-memory history
  // (splitting a long row over a larger cluster if that makes it fit)
  const int S0 = topk_cluster_size(rows, V, num_sms);
  int S = S0;
  while (S < 16 && seg_of(S) > kHistSegMax) S <<= 1;
  const bool hist = seg_of(S) <= kHistSegMax;
  if (!hist) S = S0;
  const int64_t seg_len = seg_of(S);
  {
    const cudaError_t e = hist ? allow_nonportable_clusters<topk16_hist_kernel>()
                               : allow_nonportable_clusters<topk16_kernel>();
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, static_cast<unsigned>(rows), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return hist ? cudaLaunchKernelEx(&cfg, topk16_hist_kernel, logits, V, ld, seg_len, vals, idx)
              : cudaLaunchKernelEx(&cfg, topk16_kernel, logits, V, ld, seg_len, vals, idx);
}

}  // namespace dflash2
