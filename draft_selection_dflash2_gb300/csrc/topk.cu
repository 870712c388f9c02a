// topk.cu -- per-position top-16 over bf16 logits ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector": keep the top 16 candidates of the
// drafter's own logits at every block position).
//
// Design (HBM-bound stream, 2 bytes per logit):
//   * A row is split into `S` contiguous segments, one per CTA of an S-CTA
//     thread-block cluster (S = 1 when there are enough rows to fill the GPU).
//   * A producer warp streams the segment through a ring of 16 KB shared-memory
//     stages with 1-D bulk TMA copies (cp.async.bulk, evict-first L2 policy);
//     each stage is refilled as soon as the eight consumer warps have arrived
//     on its "empty" mbarrier, so the ring never waits for a CTA barrier.
//   * Each consumer warp owns 1/8 of every stage and keeps its own running
//     top-16 (one key per lane), threshold and 64-entry candidate buffer: a
//     packed bf16x2 max over each lane's 8 logits against the warp threshold
//     rejects almost every vector; survivors become exact 64-bit keys
//     (value, -id) appended with warp ballots, folded into the warp's top-16
//     with bitonic merges whenever more than 32 are pending.
//   * At the end the eight warp lists are merged, then the S CTA lists meet in
//     distributed shared memory: CTA rank 0 reads them with ld.shared::cluster,
//     merges and writes the row's output.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace dflash2 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kStageBytes = 16384;                   // 8192 logits per stage
constexpr int kStageElems = kStageBytes / 2;
constexpr int kWarpVecs = kStageElems / 8 / kConsumerWarps;   // 128 vectors per warp per stage
constexpr int kVecPerLane = kWarpVecs / 32;                   // 4
constexpr int kStages = 4;
constexpr int kFoldAt = 32;                          // fold a warp buffer beyond this many
constexpr int kWarpCap = kFoldAt + 32 * 8;           // + one vector (8 logits) from every lane

struct TopkSmem {
  alignas(128) uint8_t stage[kStages][kStageBytes];  // 1-D bulk copies need 16-byte alignment
  uint64_t cand[kConsumerWarps][kWarpCap];
  uint64_t warp_top[kConsumerWarps][kTopK];
  uint64_t top[kTopK];
  uint64_t full_bar[kStages];
  uint64_t empty_bar[kStages];
  unsigned long long gthr;   // max over warps of their 16th-best key: a CTA-wide lower bound
  int wcount[kConsumerWarps];
  int abort_flag;
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

// Per-warp selection state; `top` is distributed (lane i < 16 holds the i-th
// best key, lanes 16..31 hold 0), `thr` is warp-uniform.
struct WarpSel {
  uint64_t top;
  uint64_t thr;
};

// Rare path, kept out of line so the streaming loop stays small in the
// instruction cache: every lane whose vector may qualify appends the keys
// above `thr` to the warp's buffer.
__device__ __noinline__ void append_vector(uint64_t* cand, int* wcount, uint4 v, uint32_t id0, uint64_t thr,
                                           bool maybe) {
  if (!maybe) return;
  for (int k = 0; k < 8; ++k) {
    const uint64_t key = make_key(lane_elem(v, k), id0 + k);
    if (key > thr) cand[atomicAdd(wcount, 1)] = key;
  }
}

// Folds the warp's pending candidates into its top-16 and publishes the new
// threshold as a CTA-wide lower bound (the CTA's 16th best is at least any
// warp's 16th best).  Whole warp.
__device__ __noinline__ void fold_warp(WarpSel& w, uint64_t* cand, int* wcount, unsigned long long* gthr, int lane) {
  __syncwarp();
  const int n = *reinterpret_cast<volatile int*>(wcount);
  for (int base = 0; base < n; base += 32)
    w.top = warp_merge_top16(w.top, base + lane < n ? cand[base + lane] : 0ull, lane);
  w.thr = __shfl_sync(0xFFFFFFFFu, w.top, kTopK - 1);
  __syncwarp();
  if (lane == 0) {
    *wcount = 0;
    atomicMax(gthr, static_cast<unsigned long long>(w.thr));
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads) topk16_kernel(const uint16_t* __restrict__ logits,
                                                          int64_t V, int64_t ld, int64_t seg_len,
                                                          float* __restrict__ vals,
                                                          int32_t* __restrict__ idx,
                                                          uint32_t* __restrict__ err) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  TopkSmem& s = *reinterpret_cast<TopkSmem*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const unsigned nrank = cluster.num_blocks();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.y;

  const int64_t seg_begin = static_cast<int64_t>(rank) * seg_len;
  const int64_t seg_end = seg_begin + seg_len < V ? seg_begin + seg_len : V;
  const int64_t n_elems = seg_end > seg_begin ? seg_end - seg_begin : 0;
  const int64_t n_vec_elems = n_elems & ~int64_t(7);          // bulk-copied part
  const int n_chunks = static_cast<int>((n_vec_elems + kStageElems - 1) / kStageElems);
  const uint16_t* seg = logits + row * ld + seg_begin;

  if (tid < kConsumerWarps) s.wcount[tid] = 0;
  if (tid == 0) {
    s.abort_flag = 0;
    s.gthr = 0ull;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full_bar[i], 1);
      mbar_init(&s.empty_bar[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &s.abort_flag;

  if (warp == kConsumerWarps) {
    // producer
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int issued = 0;
      for (int c = 0; c < n_chunks; ++c) {
        const int st = c % kStages;
        if (c >= kStages && !mbar_wait_bounded(&s.empty_bar[st], ((c / kStages) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const int64_t e0 = static_cast<int64_t>(c) * kStageElems;
        const uint32_t bytes = static_cast<uint32_t>(imin64(kStageElems, n_vec_elems - e0) * 2);
        mbar_arrive_expect_tx(&s.full_bar[st], bytes);
        bulk_g2s(s.stage[st], seg + e0, bytes, &s.full_bar[st], policy);
        issued = c + 1;
      }
      // the latest copy into every stage must land before shared memory is released
      for (int c = issued - kStages > 0 ? issued - kStages : 0; c < issued; ++c)
        mbar_wait_bounded(&s.full_bar[c % kStages], static_cast<uint32_t>(c / kStages) & 1u, err);
    }
  } else {
    // consumer warp
    WarpSel w{0ull, 0ull};
    uint64_t* cand = s.cand[warp];
    int* wcount = &s.wcount[warp];
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % kStages;
      if (!mbar_wait_bounded(&s.full_bar[st], static_cast<uint32_t>(c / kStages) & 1u, err) || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      const int64_t e0 = static_cast<int64_t>(c) * kStageElems;
      const int chunk_vecs = static_cast<int>(imin64(kStageElems, n_vec_elems - e0)) / 8;
      const uint4* sv = reinterpret_cast<const uint4*>(s.stage[st]);
      uint4 v[kVecPerLane];
      uint32_t vord[kVecPerLane];
      bool real[kVecPerLane];
#pragma unroll
      for (int h = 0; h < kVecPerLane; ++h) {
        const int vi = warp * kWarpVecs + h * 32 + lane;
        real[h] = vi < chunk_vecs;
        v[h] = real[h] ? sv[vi] : make_uint4(0u, 0u, 0u, 0u);
        vord[h] = real[h] ? bf16_order(vec_max_bits(v[h])) : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty_bar[st]);   // the stage may be refilled now
      const uint64_t g = *reinterpret_cast<volatile unsigned long long*>(&s.gthr);
      if (g > w.thr) w.thr = g;
      if ((w.thr >> 48) == 0ull) {
        // No threshold yet: the 16th largest of the 32 lane maxima is a lower
        // bound for this warp's 16th best (16 distinct elements reach it);
        // lanes without data contribute the empty key 0.
        uint32_t lm = 0u;
#pragma unroll
        for (int h = 0; h < kVecPerLane; ++h) lm = max(lm, vord[h]);
        const uint64_t sorted = warp_sort_desc(static_cast<uint64_t>(lm) << 48, lane);
        w.thr = __shfl_sync(0xFFFFFFFFu, sorted, kTopK - 1);
      }
#pragma unroll
      for (int h = 0; h < kVecPerLane; ++h) {
        const uint32_t thr_ord = static_cast<uint32_t>(w.thr >> 48);
        const bool maybe = real[h] && (thr_ord == 0u || vord[h] >= thr_ord);
        if (__ballot_sync(0xFFFFFFFFu, maybe) == 0u) continue;
        const uint32_t id0 = static_cast<uint32_t>(seg_begin + e0) + (warp * kWarpVecs + h * 32 + lane) * 8;
        append_vector(cand, wcount, v[h], id0, w.thr, maybe);
        __syncwarp();
        if (*reinterpret_cast<volatile int*>(wcount) > kFoldAt) fold_warp(w, cand, wcount, &s.gthr, lane);
      }
      // Fold whatever the chunk left at its end: the threshold then tracks the
      // 16th best seen so far and the CTA-wide bound rises with it.
      __syncwarp();
      if (*reinterpret_cast<volatile int*>(wcount) > 0) fold_warp(w, cand, wcount, &s.gthr, lane);
    }
    if (warp == 0 && !*abort_flag) {
      // ragged tail (segment length not a multiple of 8): plain loads
      const int64_t tail = n_elems - n_vec_elems;
      if (lane < tail) {
        const int64_t e = n_vec_elems + lane;
        const uint64_t key = make_key(seg[e], static_cast<uint32_t>(seg_begin + e));
        if (key > w.thr) cand[atomicAdd(wcount, 1)] = key;
      }
    }
    fold_warp(w, cand, wcount, &s.gthr, lane);
    if (lane < kTopK) s.warp_top[warp][lane] = w.top;
  }
  __syncthreads();
  if (warp == 0) {
    uint64_t acc = 0ull;
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ww += 2) {
      const uint64_t x = (lane < kTopK) ? s.warp_top[ww][lane] : s.warp_top[ww + 1][lane - kTopK];
      acc = warp_merge_top16(acc, x, lane);
    }
    if (lane < kTopK) s.top[lane] = acc;
  }

  // Merge the cluster's partial lists in distributed shared memory.
  cluster.sync();
  if (rank == 0 && warp == 0) {
    uint64_t acc = lane < kTopK ? s.top[lane] : 0ull;
    for (unsigned r = 1; r < nrank; r += 2) {
      uint64_t x = 0ull;
      const unsigned src = lane < kTopK ? r : r + 1;
      if (src < nrank) {
        const uint64_t* remote = cluster.map_shared_rank(s.top, src);
        x = remote[lane & (kTopK - 1)];
      }
      acc = warp_merge_top16(acc, x, lane);
    }
    if (lane < kTopK) {
      vals[row * kTopK + lane] = key_value(acc);
      idx[row * kTopK + lane] = key_id(acc);
    }
  }
  cluster.sync();
}

}  // namespace

int topk_cluster_size(int64_t rows, int64_t V, int num_sms) {
  // Enough CTAs for ~3 resident per SM, never a segment under one stage.
  const int64_t want = (3LL * num_sms + rows - 1) / rows;   // ~3 resident CTAs per SM
  int S = 1;
  while (S < want && S < 16) S <<= 1;
  while (S > 1 && (V + S - 1) / S < kStageElems) S >>= 1;
  return S;
}

cudaError_t launch_topk(const uint16_t* logits, int64_t rows, int64_t V, int64_t ld, float* vals,
                        int32_t* idx, uint32_t* err, int num_sms, cudaStream_t stream) {
  static bool configured = false;
  const size_t smem = sizeof(TopkSmem);
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(topk16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk16_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int S = topk_cluster_size(rows, V, num_sms);
  int64_t seg_len = (V + S - 1) / S;
  seg_len = (seg_len + 7) & ~int64_t(7);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, static_cast<unsigned>(rows), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk16_kernel, logits, V, ld, seg_len, vals, idx, err);
}

}  // namespace dflash2
