// lmhead.cu -- fused LM head + top-16: logits = hidden W^T on the tensor cores,
// reduced to each hidden row's 16 best (value, id) pairs on chip, so no logit
// ever reaches global memory.  The head produces the drafter's own logits U_t
// whose top 16 the path selector keeps ("DFlash 2: Keep Drafting Parallel",
// "A Lightweight Path Selector").
//
// lmhead_kernel (persistent, one CTA per SM):
//   CTA c owns hidden-row tile mt = c % m_tiles (128 rows) and a contiguous run
//   of vocabulary tiles (256 ids each), so the m_tiles CTAs sharing a run read
//   the same W tiles at about the same time and W streams from HBM once.
//   Pair form (an even number of row tiles): consecutive CTAs (same run, row
//   tiles 2j and 2j + 1) form a CTA pair that computes 256 x 256 tiles with
//   tcgen05.mma.cta_group::2: each CTA holds its own 128 hidden rows and half of
//   the W tile, so a 64-wide K stage brings 32 KB into each SM instead of 48 KB
//   (what each SM can take in per clock sets the pace of these GEMMs).
//   warp 0      TMA producer: 128 x 64 hidden tiles + the W tile (or, in the
//               pair form, its 128-row half) into a 4-deep (pair form: 6-deep)
//               ring with the 128-byte swizzle.  In the pair form both CTAs'
//               loads complete on the leader's stage barrier.
//   warp 1      allocates 512 TMEM columns = two 128 x 256 fp32 accumulators;
//               lane 0 issues 4 tcgen05.mma (128 x 256 x 16, or 256 x 256 x 16
//               over the pair from the leader, rank 0) per stage into the
//               current buffer and commits it when the tile's K loop is done;
//               the pair form's commits arrive in both CTAs.
//   warps 2..5  epilogue: each thread owns one hidden row (one TMEM lane) and
//               keeps its running top-16 in registers; it reads the finished
//               buffer 32 columns at a time (tcgen05.ld) and inserts the rare
//               logits above its 16th best, then hands the buffer back (to the
//               leader, in the pair form), so the epilogue of tile i overlaps
//               the MMAs of tile i + 1.
//   At the end each thread writes its list as 16 order-preserving 64-bit keys
//   (fp32 value, -id) to the workspace [M, n_runs, 16].
//   With the context gate folded in, W_H's 256 rows are one more "vocabulary"
//   tile after the last (0.17% more products at V = 151936): its epilogue
//   writes H = sigmoid(acc + b_H) for the tile's rows instead of ranking them.
// lmhead_merge_kernel: one warp per row folds the n_runs partial lists into the
// final top-16 (value descending, lowest id on ties).
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace dflash2 {
namespace {

constexpr int kLmBN = 256;
constexpr int kLmThreads = 192;
constexpr int kLmABytes = 128 * kTileRowBytes;                 // 16 KB
constexpr int kLmMaxStages = 6;
constexpr uint32_t kLmTmemCols = 2 * kLmBN;                    // double-buffered accumulator

// W rows per CTA, stage size and ring depth of each form
template <bool kPair>
struct LmForm {
  static constexpr int kWRows = kPair ? kLmBN / 2 : kLmBN;
  static constexpr int kStageBytes = kLmABytes + kWRows * kTileRowBytes;
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr uint32_t kIdesc = umma_idesc_bf16(kPair ? 256 : 128, kLmBN);
};

struct LmSmem {
  uint64_t full[kLmMaxStages];     // pair form: the leader's count both CTAs' bytes
  uint64_t empty[kLmMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];              // pair form: the leader's count both CTAs' epilogue warps
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of this CTA's shared variable at `p` in the shared window of cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// Pair form: the box at (x, y) into this CTA's shared memory, completing tx
// bytes on the barrier at cluster address `bar` (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// Pair form: D[tmem] (+)= A B^T over both CTAs' operands at the same shared offsets.
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair form: arrives once on `bar` in both CTAs when the pair's MMAs so far are complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Pair form: arrives once on this CTA's `bar` when the pair's MMAs so far are complete.
__device__ __forceinline__ void umma_commit_pair_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

// Arrives once on the barrier at cluster address `bar` (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

template <bool kPair>
__device__ __forceinline__ void lm_tmem_alloc(uint32_t* dst) {
  if constexpr (kPair) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(kLmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    tmem_alloc(dst, kLmTmemCols);
    tmem_relinquish();
  }
}

template <bool kPair>
__device__ __forceinline__ void lm_tmem_dealloc(uint32_t taddr) {
  if constexpr (kPair)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kLmTmemCols) : "memory");
  else
    tmem_dealloc(taddr, kLmTmemCols);
}

// Order-preserving 64-bit key of an fp32 logit and its id: larger key ranks
// first (value descending, then id ascending); 0 is "empty".
__device__ __forceinline__ uint64_t logit_key(float v, int32_t id) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;                       // -0 == +0
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~static_cast<uint32_t>(id));
}

__device__ __forceinline__ float logit_key_value(uint64_t k) {
  const uint32_t ord = static_cast<uint32_t>(k >> 32);
  const uint32_t b = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(b);
}

template <bool kPair>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmH, int M, int64_t V, int d, int m_tiles, int n_tiles,
                  int n_vocab_tiles, int tiles_per_run, int n_runs, uint64_t* __restrict__ partial,
                  float* __restrict__ gate, const float* __restrict__ b_H, uint32_t* __restrict__ err) {
  using F = LmForm<kPair>;
  constexpr int S = F::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = align_smem<1024>(smem_raw);
  LmSmem& s = *reinterpret_cast<LmSmem*>(ring + S * F::kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x % m_tiles;
  const int run = blockIdx.x / m_tiles;
  const int nt0 = run * tiles_per_run;
  const int nt1 = min(n_tiles, nt0 + tiles_per_run);
  const int ntiles = max(0, nt1 - nt0);
  const int nk = d / kBK;
  // pair form: rank 0 leads (issues the MMAs); rank r holds W rows [r * 128, +128) of each tile
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], kPair ? 8 : 4);   // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (gate) tma_prefetch_desc(&tmH);
  }
  if (warp == 1) lm_tmem_alloc<kPair>(&s.tmem);
  tc_fence_before();
  __syncthreads();
  if (kPair) {
    // both CTAs' barriers and TMEM exist before any remote arrival or pair MMA
    cluster_arrive();
    cluster_wait();
  }
  tc_fence_after();
  const uint32_t tmem = s.tmem;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_last();    // hidden rows: reused by every tile
      // W tiles are read by the m_tiles CTAs sharing a run at slightly different
      // times: normal priority keeps them in L2 until the last of those reads
      uint64_t pol_b;
      asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_b));
      int it = 0, issued = 0;
      for (int i = 0; i < ntiles && !*abort_flag; ++i) {
        const bool gate_tile = nt0 + i == n_vocab_tiles;   // W_H (only when folded in)
        const CUtensorMap* tw = gate_tile ? &tmH : &tmB;
        const int wrow = (gate_tile ? 0 : (nt0 + i) * kLmBN) + static_cast<int>(rank) * F::kWRows;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % S;
          if (it >= S && !mbar_wait_bounded(&s.empty[st], ((it / S) - 1) & 1, err)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* a_dst = ring + st * F::kStageBytes;
          if constexpr (kPair) {
            // both CTAs' halves complete on the leader's barrier, which expects them all
            if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * F::kStageBytes);
            const uint32_t bar = cluster_addr(&s.full[st], 0);
            tma_load_2d_pair(a_dst, &tmA, kb * kBK, mt * 128, bar, pol_a);
            tma_load_2d_pair(a_dst + kLmABytes, tw, kb * kBK, wrow, bar, gate_tile ? pol_a : pol_b);
          } else {
            mbar_arrive_expect_tx(&s.full[st], F::kStageBytes);
            tma_load_2d(a_dst, &tmA, kb * kBK, mt * 128, &s.full[st], pol_a);
            tma_load_2d(a_dst + kLmABytes, tw, kb * kBK, wrow, &s.full[st], gate_tile ? pol_a : pol_b);
          }
          issued = it + 1;
        }
      }
      // before this CTA may exit: its own copies have landed (the leader's
      // barrier saw them) and the pair's MMAs are done with every stage
      for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j) {
        if (!kPair || leader) mbar_wait_bounded(&s.full[j % S], (j / S) & 1, err);
        mbar_wait_bounded(&s.empty[j % S], (j / S) & 1, err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int it = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int buf = i & 1;
        if (i >= 2 && !mbar_wait_bounded(&s.tempty[buf], ((i >> 1) - 1) & 1, err)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * kLmBN;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int st = it % S;
          if (!mbar_wait_bounded(&s.full[st], (it / S) & 1, err) || *abort_flag) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(ring + st * F::kStageBytes);
          const uint32_t b_base = a_base + kLmABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = umma_desc_sw128(a_base + k * 32), bd = umma_desc_sw128(b_base + k * 32);
            if constexpr (kPair)
              umma_bf16_pair(acc, ad, bd, F::kIdesc, (kb | k) != 0 ? 1u : 0u);
            else
              umma_bf16(acc, ad, bd, F::kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          if constexpr (kPair)
            umma_commit_pair(&s.empty[st]);
          else
            umma_commit(&s.empty[st]);
        }
        if constexpr (kPair)
          umma_commit_pair(&s.tfull[buf]);
        else
          umma_commit(&s.tfull[buf]);
        if (!ok) break;
      }
    }
  } else {
    // epilogue: one hidden row per thread
    const int q = warp & 3;
    const int row = mt * 128 + q * 32 + lane;
    const bool row_ok = row < M;
    // the leader's MMA waits for every epilogue warp of the pair before reusing a buffer
    const uint32_t tempty0 = kPair ? cluster_addr(&s.tempty[0], 0) : 0u;
    const uint32_t tempty1 = kPair ? cluster_addr(&s.tempty[1], 0) : 0u;
    float val[kTopK];
    int32_t ids[kTopK];
#pragma unroll
    for (int k = 0; k < kTopK; ++k) {
      val[k] = -INFINITY;
      ids[k] = 0x7FFFFFFF;
    }
    for (int i = 0; i < ntiles; ++i) {
      const int buf = i & 1;
      if (!mbar_wait_bounded(&s.tfull[buf], (i >> 1) & 1, err) || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const bool gate_tile = nt0 + i == n_vocab_tiles;
      const int64_t id_base = static_cast<int64_t>(nt0 + i) * kLmBN;
#pragma unroll 1
      for (int c = 0; c < kLmBN / 32; ++c) {
        float v[32];
        tmem_ld_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kLmBN + c * 32, v);
        tmem_ld_wait();
        if (c == kLmBN / 32 - 1) {
          // the buffer is read out: hand it back to the MMA issuer
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair)
              mbar_arrive_cluster(buf ? tempty1 : tempty0);
            else
              mbar_arrive(&s.tempty[buf]);
          }
        }
        if (!row_ok) continue;
        if (gate_tile) {
          // gate tile: H[row, c] = sigmoid(acc + b_H[c])
          float* dst = gate + static_cast<int64_t>(row) * kEmbed + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o[u] = 1.0f / (1.0f + expf(-(v[j + u] + (b_H ? b_H[c * 32 + j + u] : 0.0f))));
            *reinterpret_cast<float4*>(dst + j) = make_float4(o[0], o[1], o[2], o[3]);
          }
          continue;
        }
        const int64_t id0 = id_base + c * 32;
        // the common case (nothing above the row's 16th best) costs one compare
        // per logit; the sorted insertion stays a compact loop
        float m = v[0];
#pragma unroll
        for (int j = 1; j < 32; ++j) m = fmaxf(m, v[j]);
        if (m > val[kTopK - 1]) {
#pragma unroll 1
          for (int j = 0; j < 32; ++j) {
            const float x = v[j];
            if (x > val[kTopK - 1] && id0 + j < V) {
              // ids arrive in increasing order, so an equal value (larger id)
              // never displaces an existing entry
              float cv = x;
              int32_t ci = static_cast<int32_t>(id0 + j);
#pragma unroll
              for (int k = 0; k < kTopK; ++k) {
                const bool sw = cv > val[k];
                const float tv = val[k];
                const int32_t ti = ids[k];
                val[k] = sw ? cv : tv;
                ids[k] = sw ? ci : ti;
                cv = sw ? tv : cv;
                ci = sw ? ti : ci;
              }
            }
          }
        }
      }
    }
    if (row_ok) {
      uint64_t* dst = partial + (static_cast<int64_t>(row) * n_runs + run) * kTopK;
#pragma unroll
      for (int k = 0; k < kTopK; ++k) dst[k] = (ids[k] == 0x7FFFFFFF) ? 0ull : logit_key(val[k], ids[k]);
    }
  }

  __syncthreads();
  if (warp == 1 && leader) {
    if (lane == 0) {
      if constexpr (kPair)
        umma_commit_pair_local(&s.drain);
      else
        umma_commit(&s.drain);
      mbar_wait_bounded(&s.drain, 0, err);
    }
    __syncwarp();
  }
  if (kPair) {
    // the leader's MMAs are complete and every remote arrival has landed
    // before either CTA frees its TMEM or leaves
    tc_fence_before();
    cluster_arrive();
    cluster_wait();
  }
  if (warp == 1) {
    tc_fence_after();
    lm_tmem_dealloc<kPair>(tmem);
  }
}

// One warp per row: the top-16 of the row's n_runs partial lists.
__global__ void lmhead_merge_kernel(const uint64_t* __restrict__ partial, int M, int n_runs,
                                    float* __restrict__ vals, int32_t* __restrict__ idx) {
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint64_t* src = partial + static_cast<int64_t>(row) * n_runs * kTopK;
  const int n = n_runs * kTopK;
  uint64_t top = 0ull;
  for (int base = 0; base < n; base += 32) top = warp_merge_top16(top, base + lane < n ? src[base + lane] : 0ull, lane);
  if (lane < kTopK) {
    vals[static_cast<int64_t>(row) * kTopK + lane] = logit_key_value(top);
    idx[static_cast<int64_t>(row) * kTopK + lane] = static_cast<int32_t>(~static_cast<uint32_t>(top));
  }
}

struct LmPlan {
  int m_tiles, n_tiles, n_runs, tiles_per_run, grid;
};

LmPlan lm_plan(int64_t M, int64_t V, int num_sms) {
  LmPlan p;
  p.m_tiles = static_cast<int>((M + 127) / 128);
  p.n_tiles = static_cast<int>((V + kLmBN - 1) / kLmBN);
  int runs = num_sms / p.m_tiles;
  if (runs < 1) runs = 1;
  if (runs > p.n_tiles) runs = p.n_tiles;
  p.tiles_per_run = (p.n_tiles + runs - 1) / runs;
  p.n_runs = (p.n_tiles + p.tiles_per_run - 1) / p.tiles_per_run;
  p.grid = p.m_tiles * p.n_runs;
  return p;
}

}  // namespace

// Fixed scratch for dflash2_lmhead_topk_noalloc: the partial lists live in
// this file-scope device array instead of a caller-provided workspace.  Every
// GPU that loads the library holds it until the process exits.
static __device__ __align__(256) uint8_t g_lmhead_scratch[kLmheadNoAllocScratchBytes];

cudaError_t lmhead_noalloc_scratch(int device, void** ptr) {
  // The array's device address, looked up once per device with that device
  // current (its host-side name is only a stand-in for the symbol).
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return e;
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
    if (prev != device) {
      const cudaError_t e2 = cudaSetDevice(prev);
      if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return e;
    addr[device] = p;
  }
  *ptr = addr[device];
  return cudaSuccess;
}

size_t lmhead_workspace_bytes(int64_t M, int64_t V, int64_t d, int num_sms) {
  (void)d;
  // covers the plain head and the head with the gate tile folded in
  const LmPlan p = lm_plan(M, V, num_sms), pg = lm_plan(M, V + kLmBN, num_sms);
  const int n_runs = p.n_runs > pg.n_runs ? p.n_runs : pg.n_runs;
  return static_cast<size_t>(M) * n_runs * kTopK * sizeof(uint64_t);
}

namespace {

template <bool kPair>
cudaError_t launch_lmhead_form(const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H, const float* b_H,
                               int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx, float* gate,
                               void* workspace, int num_sms, uint32_t* err, cudaStream_t stream) {
  using F = LmForm<kPair>;
  const int n_vocab_tiles = static_cast<int>((V + kLmBN - 1) / kLmBN);
  const int64_t Vt = gate ? V + kLmBN : V;
  const size_t smem = 1024 + F::kStages * F::kStageBytes + sizeof(LmSmem);
  {
    const cudaError_t e = set_smem_limit<lmhead_kernel<kPair>>(smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kLmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2u : 1u;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int slots = num_sms;
  if (kPair) {
    // the runs are sized to the pairs that can be resident at once on this device
    static std::mutex mu;
    static int resident[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (resident[dev] == 0) {
      cfg.gridDim = dim3(2, 1, 1);
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, lmhead_kernel<kPair>, &cfg);
      if (e != cudaSuccess) return e;
      resident[dev] = n > 0 ? n : 1;
    }
    slots = 2 * resident[dev];
  }
  const LmPlan p = lm_plan(M, Vt, slots);
  CUtensorMap ta, tb, th;
  if (!make_tmap_bf16_2d(&ta, hidden, M, d, d, 128) || !make_tmap_bf16_2d(&tb, W, V, d, d, F::kWRows))
    return cudaErrorInvalidValue;
  if (gate) {
    if (!make_tmap_bf16_2d(&th, W_H, kEmbed, d, d, F::kWRows)) return cudaErrorInvalidValue;
  } else {
    th = tb;
  }
  uint64_t* partial = static_cast<uint64_t*>(workspace);
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid), 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, lmhead_kernel<kPair>, ta, tb, th, static_cast<int>(M), V,
                                     static_cast<int>(d), p.m_tiles, p.n_tiles, n_vocab_tiles, p.tiles_per_run,
                                     p.n_runs, partial, gate, b_H, err);
  if (e != cudaSuccess) return e;
  const int rows_per_block = 8;
  lmhead_merge_kernel<<<static_cast<unsigned>((M + rows_per_block - 1) / rows_per_block), 32 * rows_per_block, 0,
                        stream>>>(partial, static_cast<int>(M), p.n_runs, vals, idx);
  return cudaGetLastError();
}

cudaError_t launch_lmhead(const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H, const float* b_H,
                          int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx, float* gate, void* workspace,
                          int num_sms, uint32_t* err, cudaStream_t stream) {
  if (d % kBK != 0 || M > 0x7FFFFFFF || d > 0x7FFFFFFF) return cudaErrorInvalidValue;
  // an even number of 128-row tiles pairs up consecutive row tiles
  const int64_t m_tiles = (M + 127) / 128;
  if (m_tiles % 2 == 0)
    return launch_lmhead_form<true>(hidden, W, W_H, b_H, M, V, d, vals, idx, gate, workspace, num_sms, err, stream);
  return launch_lmhead_form<false>(hidden, W, W_H, b_H, M, V, d, vals, idx, gate, workspace, num_sms, err, stream);
}

}  // namespace

cudaError_t launch_lmhead_topk(const uint16_t* hidden, const uint16_t* W, int64_t M, int64_t V,
                               int64_t d, float* vals, int32_t* idx, void* workspace, int num_sms,
                               uint32_t* err, cudaStream_t stream) {
  return launch_lmhead(hidden, W, nullptr, nullptr, M, V, d, vals, idx, nullptr, workspace, num_sms, err, stream);
}

cudaError_t launch_lmhead_topk_gate(const uint16_t* hidden, const uint16_t* W, const uint16_t* W_H,
                                    const float* b_H, int64_t M, int64_t V, int64_t d, float* vals, int32_t* idx,
                                    float* gate, void* workspace, int num_sms, uint32_t* err,
                                    cudaStream_t stream) {
  return launch_lmhead(hidden, W, W_H, b_H, M, V, d, vals, idx, gate, workspace, num_sms, err, stream);
}

}  // namespace dflash2
