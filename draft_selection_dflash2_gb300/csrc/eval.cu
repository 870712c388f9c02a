// eval.cu -- the selector evaluation of Table 1 ("DFlash 2: Keep Drafting
// Parallel", "The Right Tokens Are Already There"): per-position recall of the
// top-1 and of the top-16 candidates, conditioned on every earlier position
// being right under the same rule, and the acceptance lengths they imply (the
// verifier's next token included).
//
// A CTA takes chunks of 256 consecutive sequences (a persistent grid of 8
// CTAs per SM strides over them).  Phase 1 streams their candidate rows
// (64 B each) with four lanes per row, each lane loading 16 B, and stores one
// flag byte per row in shared memory: bit 0 = slot 0 holds the true token,
// bit 1 = one of the 16 slots does.  Phase 2 gives each sequence one thread,
// which counts its leading bit-0 rows (n1) and leading bit-1 rows (n16):
// accept1 = 1 + n1, accept16 = 1 + n16.  Position t is reached under a rule by
// every sequence whose leading count is >= t and hit there by those whose count
// is >= t + 1, so the [L, 4] counts are suffix sums of the n1 / n16 histograms;
// each CTA keeps its histograms in shared memory over all its chunks and adds
// their suffix sums to the global table with one 64-bit atomic per entry.
#include "common.cuh"
#include "launch.h"

namespace dflash2 {
namespace {

constexpr int kEvalThreads = 256;            // = sequences per CTA
constexpr int kEvalMaxL = 64;
constexpr int kEvalRowsPerPass = kEvalThreads / 4;
constexpr int kEvalUnroll = 8;
constexpr int kEvalCtasPerSm = 8;            // 2048 threads per SM

__global__ void selector_eval_zero(unsigned long long* counts, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) counts[i] = 0ull;
}

// kVec: cand_idx is 16-byte aligned (every 64-byte row then is too)
template <bool kVec>
__global__ void __launch_bounds__(kEvalThreads)
    selector_eval_kernel(const int32_t* __restrict__ gt, const int32_t* __restrict__ cand_idx, int64_t B, int L,
                         int32_t* __restrict__ accept1, int32_t* __restrict__ accept16,
                         unsigned long long* __restrict__ counts) {
  __shared__ uint8_t flags[kEvalThreads * kEvalMaxL];
  __shared__ unsigned int hist[2][kEvalMaxL + 1];
  const int tid = threadIdx.x, lane = tid & 31, sub = tid & 3, grp = tid >> 2;
  for (int i = tid; i < 2 * (kEvalMaxL + 1); i += kEvalThreads) (&hist[0][0])[i] = 0u;

  // persistent: chunks of 256 sequences strided over the grid
  for (int64_t s0 = static_cast<int64_t>(blockIdx.x) * kEvalThreads; s0 < B;
       s0 += static_cast<int64_t>(gridDim.x) * kEvalThreads) {
    const int nseq = static_cast<int>(B - s0 < kEvalThreads ? B - s0 : kEvalThreads);
    const int nrows = nseq * L;
    const int64_t row0 = s0 * L;

    // phase 1: flag bytes, kEvalUnroll row groups in flight per thread
    for (int base = 0; base < nrows; base += kEvalRowsPerPass * kEvalUnroll) {
      int4 v[kEvalUnroll];
      int32_t g[kEvalUnroll];
#pragma unroll
      for (int u = 0; u < kEvalUnroll; ++u) {
        const int r = base + u * kEvalRowsPerPass + grp;
        v[u] = make_int4(0, 0, 0, 0);
        g[u] = 0;
        if (r < nrows) {
          const int32_t* row = cand_idx + (row0 + r) * kTopK + sub * 4;
          if constexpr (kVec) {
            v[u] = __ldcs(reinterpret_cast<const int4*>(row));
          } else {
            v[u] = make_int4(__ldcs(row), __ldcs(row + 1), __ldcs(row + 2), __ldcs(row + 3));
          }
          g[u] = __ldcs(gt + row0 + r);
        }
      }
#pragma unroll
      for (int u = 0; u < kEvalUnroll; ++u) {
        const int r = base + u * kEvalRowsPerPass + grp;
        const bool first = v[u].x == g[u];
        const bool any4 = first || v[u].y == g[u] || v[u].z == g[u] || v[u].w == g[u];
        // the four lanes of a row are lanes 4q .. 4q + 3 of one warp; lane 4q holds slots 0..3
        const unsigned m = __ballot_sync(0xFFFFFFFFu, any4);
        const unsigned f = __ballot_sync(0xFFFFFFFFu, first);
        const int q = lane & ~3;
        const bool any = ((m >> q) & 0xFu) != 0u;
        const bool top = ((f >> q) & 1u) != 0u;
        if (sub == 0 && r < nrows) flags[r] = static_cast<uint8_t>((top ? 1u : 0u) | (any ? 2u : 0u));
      }
    }
    __syncthreads();

    // phase 2: leading hits per sequence; lanes with equal counts add to the
    // histogram once (most sequences of a warp share a count)
    int n1 = -1, n16 = -1;
    if (tid < nseq) {
      const uint8_t* fr = flags + tid * L;
      n1 = 0;
      n16 = 0;
      while (n16 < L && (fr[n16] & 2u)) ++n16;
      while (n1 < n16 && (fr[n1] & 1u)) ++n1;      // slot 0 is one of the 16: n1 <= n16
      accept1[s0 + tid] = 1 + n1;
      accept16[s0 + tid] = 1 + n16;
    }
    const unsigned same1 = __match_any_sync(0xFFFFFFFFu, n1);
    const unsigned same16 = __match_any_sync(0xFFFFFFFFu, n16);
    if (n1 >= 0 && (same1 & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[0][n1], __popc(same1));
    if (n16 >= 0 && (same16 & ((1u << lane) - 1u)) == 0u) atomicAdd(&hist[1][n16], __popc(same16));
    __syncthreads();   // the next chunk's phase 1 overwrites the flags
  }

  // counts[t] = {#(n1 >= t), #(n1 >= t + 1), #(n16 >= t), #(n16 >= t + 1)}
  if (tid < L) {
    unsigned int a1 = 0u, a16 = 0u;
    for (int n = tid + 1; n <= L; ++n) {
      a1 += hist[0][n];
      a16 += hist[1][n];
    }
    const unsigned int r1 = a1 + hist[0][tid], r16 = a16 + hist[1][tid];
    unsigned long long* c = counts + tid * 4;
    if (r1) atomicAdd(c + 0, static_cast<unsigned long long>(r1));
    if (a1) atomicAdd(c + 1, static_cast<unsigned long long>(a1));
    if (r16) atomicAdd(c + 2, static_cast<unsigned long long>(r16));
    if (a16) atomicAdd(c + 3, static_cast<unsigned long long>(a16));
  }
}

}  // namespace

cudaError_t launch_selector_eval(const int32_t* gt, const int32_t* cand_idx, int64_t B, int64_t L, int32_t* accept1,
                                 int32_t* accept16, int64_t* counts, int num_sms, cudaStream_t stream) {
  if (L > kEvalMaxL) return cudaErrorInvalidValue;
  unsigned long long* cnt = reinterpret_cast<unsigned long long*>(counts);
  selector_eval_zero<<<1, kEvalThreads, 0, stream>>>(cnt, L * 4);
  if (B == 0) return cudaGetLastError();
  const int64_t chunks = (B + kEvalThreads - 1) / kEvalThreads;
  const unsigned grid = static_cast<unsigned>(chunks < int64_t(num_sms) * kEvalCtasPerSm ? chunks
                                                                                          : int64_t(num_sms) * kEvalCtasPerSm);
  if ((reinterpret_cast<uintptr_t>(cand_idx) & 15u) == 0u)
    selector_eval_kernel<true><<<grid, kEvalThreads, 0, stream>>>(gt, cand_idx, B, static_cast<int>(L), accept1,
                                                                  accept16, cnt);
  else
    selector_eval_kernel<false><<<grid, kEvalThreads, 0, stream>>>(gt, cand_idx, B, static_cast<int>(L), accept1,
                                                                   accept16, cnt);
  return cudaGetLastError();
}

}  // namespace dflash2
