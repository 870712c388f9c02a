// topk.cu -- per-position top-16 over bf16 logits ("DFlash 2: Keep Drafting
// Parallel", "A Lightweight Path Selector": keep the top 16 candidates of the
// drafter's own logits at every block position).
//
// Design (HBM-bound stream, 2 bytes per logit):
//   * A row is split into `S` contiguous segments, one per CTA of an S-CTA
//     thread-block cluster (S = 1 when there are enough rows to fill the GPU).
//   * Each CTA streams its segment through a ring of shared-memory stages with
//     1-D bulk TMA copies (cp.async.bulk, evict-first L2 policy), so global
//     loads are 8 KB transactions issued by one thread.
//   * Every thread scans 16 logits per stage.  A packed bf16x2 max over those
//     16 against the CTA's running 16th-best value rejects almost every group
//     in ~10 instructions; survivors are turned into exact 64-bit keys
//     (value, -id) and appended to a shared candidate buffer.
//   * When the buffer passes 64 entries (and at the end) the warps fold it into
//     the running top-16 with warp-level bitonic merges and raise the threshold.
//   * The S partial lists meet in distributed shared memory: CTA rank 0 reads
//     them with ld.shared::cluster, merges and writes the row's output.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

namespace dflash2 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStageBytes = 16384;                   // 8192 logits per stage
constexpr int kStageElems = kStageBytes / 2;
constexpr int kVecPerThread = kStageElems / 8 / kThreads;   // 4 x 16-byte vectors
constexpr int kStages = 4;
constexpr int kCompactAt = 64;                       // fold the buffer beyond this many
constexpr int kCandCap = 512 + kCompactAt;           // overflow -> the chunk is rescanned
constexpr int kRescanVecs = 64;                      // vectors per rescan slice (512 logits)

struct TopkSmem {
  alignas(128) uint8_t stage[kStages][kStageBytes];   // 1-D bulk copies need 16-byte alignment
  uint64_t cand[kCandCap];
  uint64_t top[kTopK];        // running top-16, descending
  uint64_t warp_top[kWarps][kTopK];
  uint64_t full_bar[kStages];
  uint64_t thr_key;           // top[15] (0 while fewer than 16 seen)
  unsigned long long init_thr;  // lower bound used for a chunk that starts with no threshold
  int count;
  int count0;                 // count at the start of the current chunk
  int overflow;
};

// Folds cand[0..n) into s.top using every warp; leaves s.thr_key updated and
// s.count = 0.  Must be called by all threads of the CTA (contains __syncthreads).
__device__ void fold_candidates(TopkSmem& s, int n, int warp, int lane) {
  if (n <= 32) {
    if (warp == 0) {
      uint64_t top = lane < kTopK ? s.top[lane] : 0ull;
      const uint64_t x = lane < n ? s.cand[lane] : 0ull;
      top = warp_merge_top16(top, x, lane);
      if (lane < kTopK) s.top[lane] = top;
      if (lane == kTopK - 1) s.thr_key = top;
      if (lane == 0) s.count = 0;
    }
    __syncthreads();
    return;
  }
  uint64_t top = 0ull;
  for (int base = warp * 32; base < n; base += kWarps * 32) {
    const int i = base + lane;
    top = warp_merge_top16(top, i < n ? s.cand[i] : 0ull, lane);
  }
  if (lane < kTopK) s.warp_top[warp][lane] = top;
  __syncthreads();
  if (warp == 0) {
    uint64_t acc = lane < kTopK ? s.top[lane] : 0ull;
#pragma unroll
    for (int w = 0; w < kWarps; w += 2) {
      const uint64_t x = (lane < kTopK) ? s.warp_top[w][lane] : s.warp_top[w + 1][lane - kTopK];
      acc = warp_merge_top16(acc, x, lane);
    }
    if (lane < kTopK) s.top[lane] = acc;
    if (lane == kTopK - 1) s.thr_key = acc;
    if (lane == 0) s.count = 0;
  }
  __syncthreads();
}

__device__ __forceinline__ void push_candidate(TopkSmem& s, uint64_t key) {
  const int slot = atomicAdd(&s.count, 1);
  if (slot < kCandCap)
    s.cand[slot] = key;
  else
    s.overflow = 1;   // the chunk is rolled back and rescanned in slices
}

// Examines 8 logits (one 16-byte vector) whose first id is `id0`.
__device__ __forceinline__ void scan_vector(TopkSmem& s, uint4 v, uint32_t id0, uint64_t thr) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t bits = h ? (w[q] >> 16) : (w[q] & 0xFFFFu);
      const uint64_t key = make_key(bits, id0 + 2 * q + h);
      if (key > thr) push_candidate(s, key);
    }
  }
}

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

  if (tid < kTopK) s.top[tid] = 0ull;
  if (tid == 0) {
    s.count = 0;
    s.count0 = 0;
    s.overflow = 0;
    s.thr_key = 0ull;
    s.init_thr = 0ull;
    for (int i = 0; i < kStages; ++i) mbar_init(&s.full_bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t policy = 0;
  if (tid == 0) {
    policy = l2_policy_evict_first();
    for (int c = 0; c < kStages && c < n_chunks; ++c) {
      const int64_t e0 = static_cast<int64_t>(c) * kStageElems;
      const uint32_t bytes = static_cast<uint32_t>(imin64(kStageElems, n_vec_elems - e0) * 2);
      mbar_arrive_expect_tx(&s.full_bar[c], bytes);
      bulk_g2s(s.stage[c], seg + e0, bytes, &s.full_bar[c], policy);
    }
  }

  int aborted_at = -1;   // CTA-uniform
  for (int c = 0; c < n_chunks; ++c) {
    const int st = c % kStages;
    const uint32_t parity = static_cast<uint32_t>(c / kStages) & 1u;
    const bool ok = mbar_wait_bounded(&s.full_bar[st], parity, err);
    if (__syncthreads_or(!ok)) {
      aborted_at = c;
      break;
    }
    const int64_t e0 = static_cast<int64_t>(c) * kStageElems;
    const int chunk_elems = static_cast<int>(imin64(kStageElems, n_vec_elems - e0));
    const uint32_t id_base = static_cast<uint32_t>(seg_begin + e0);
    const uint4* sv = reinterpret_cast<const uint4*>(s.stage[st]);
    uint4 v[kVecPerThread];
    uint32_t vmax[kVecPerThread];
#pragma unroll
    for (int h = 0; h < kVecPerThread; ++h) {
      const int vi = tid + h * kThreads;
      v[h] = (vi * 8 < chunk_elems) ? sv[vi] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
      vmax[h] = vec_max_bits(v[h]);
    }
    uint64_t thr = s.thr_key;
    if ((thr >> 48) == 0ull) {
      // Threshold still empty: a lower bound for this CTA's 16th best is the
      // 16th largest of any warp's 32 per-thread maxima (16 distinct elements
      // reach it).  Take the largest such bound over the warps.
      // Threads without data contribute the empty key 0.
      uint32_t tmax = 0;
#pragma unroll
      for (int h = 0; h < kVecPerThread; ++h)
        if ((tid + h * kThreads) * 8 < chunk_elems) tmax = max(tmax, bf16_order(vmax[h]));
      const uint64_t sorted = warp_sort_desc(static_cast<uint64_t>(tmax) << 48, lane);
      if (lane == kTopK - 1) atomicMax(&s.init_thr, static_cast<unsigned long long>(sorted));
      if (tid == 0) s.count0 = s.count;
      __syncthreads();
      thr = s.init_thr;
      __syncthreads();
      if (tid == 0) s.init_thr = 0ull;
    } else if (tid == 0) {
      s.count0 = s.count;
    }
    // elements equal to the bound keep qualifying (its id field is 0)
    const bool exact_only = (thr >> 48) == 0ull;
    const uint32_t thr_ord = static_cast<uint32_t>(thr >> 48);
#pragma unroll
    for (int h = 0; h < kVecPerThread; ++h) {
      const int vi = tid + h * kThreads;
      if (vi * 8 < chunk_elems && (exact_only || bf16_order(vmax[h]) >= thr_ord))
        scan_vector(s, v[h], id_base + vi * 8, thr);
    }
    __syncthreads();   // stage consumed, all pushes visible
    if (s.overflow) {
      // Roll the chunk back (drop what it pushed), then rescan it in slices of
      // 512 logits with a fold after each slice, so no slice can overflow.
      const int n0 = s.count0;
      __syncthreads();
      fold_candidates(s, n0, warp, lane);
      if (tid == 0) s.overflow = 0;
      const int nvec = chunk_elems / 8;
      for (int sl = 0; sl < nvec; sl += kRescanVecs) {
        const uint64_t t2 = s.thr_key;
        if (tid < kRescanVecs && sl + tid < nvec) scan_vector(s, sv[sl + tid], id_base + (sl + tid) * 8, t2);
        __syncthreads();
        fold_candidates(s, s.count, warp, lane);
      }
    }
    if (tid == 0 && c + kStages < n_chunks) {
      const int64_t e1 = static_cast<int64_t>(c + kStages) * kStageElems;
      const uint32_t bytes = static_cast<uint32_t>(imin64(kStageElems, n_vec_elems - e1) * 2);
      mbar_arrive_expect_tx(&s.full_bar[st], bytes);
      bulk_g2s(s.stage[st], seg + e1, bytes, &s.full_bar[st], policy);
    }
    const int n = s.count;
    if (n > kCompactAt) fold_candidates(s, n, warp, lane);
  }

  if (aborted_at >= 0) {
    // Let the copies still in flight land before the CTA's shared memory goes away.
    if (tid == 0) {
      for (int c = aborted_at; c < n_chunks && c < aborted_at + kStages; ++c)
        mbar_wait_bounded(&s.full_bar[c % kStages], static_cast<uint32_t>(c / kStages) & 1u, err);
    }
  } else {
    // Ragged tail (segment length not a multiple of 8): plain loads.
    const int64_t tail = n_elems - n_vec_elems;
    if (tid < tail) {
      const int64_t e = n_vec_elems + tid;
      const uint64_t key = make_key(seg[e], static_cast<uint32_t>(seg_begin + e));
      if (key > s.thr_key) push_candidate(s, key);
    }
    __syncthreads();
    const int n = s.count;
    if (n > 0) fold_candidates(s, n, warp, lane);
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
  const int64_t want = (3LL * num_sms + rows - 1) / rows;
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
