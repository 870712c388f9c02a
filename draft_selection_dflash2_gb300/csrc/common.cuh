// common.cuh -- device helpers shared by the DFlash 2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash2.h"

namespace dflash2 {

constexpr int kTopK = 16;
constexpr int kEmbed = 256;   // r: width of the selector embeddings and the gate

// Upper bound on any bounded device wait, in nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// error word
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ int32_t clamp_token(int32_t id, int64_t V, uint32_t* err) {
  if (id < 0 || id >= V) {
    raise_error(err, DFLASH2_DEVERR_BAD_TOKEN);
    return id < 0 ? 0 : static_cast<int32_t>(V - 1);
  }
  return id;
}

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }

// Programmatic dependent launch.  pdl_wait blocks until the grid this one was
// launched after has completed and its writes are visible (a no-op when the
// launch did not allow programmatic serialization), so it comes before a
// kernel's first global access; pdl_launch_dependents lets the next grid in
// the stream be scheduled (its CTAs run their own prologue and then wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers and bulk (TMA) copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Rounds a dynamic shared-memory base up to kAlign bytes by pointer arithmetic
// on the shared array itself: the compiler then still knows that the result,
// and every pointer derived from it, addresses shared memory, and emits
// shared-memory instructions for the accesses (a round trip through an
// integer would turn each of them into a slower generic access).
template <int kAlign>
__device__ __forceinline__ uint8_t* align_smem(uint8_t* base) {
  return base + ((kAlign - (smem_addr(base) & (kAlign - 1))) & (kAlign - 1));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after limit_ns.
// Returns false (and raises DFLASH2_DEVERR_TIMEOUT) if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - start > limit_ns) {
      raise_error(err, DFLASH2_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Waits until the word at `flag` (written by another CTA) reaches `value`,
// giving up after limit_ns.  Returns false (and raises DFLASH2_DEVERR_TIMEOUT)
// if it gave up.
__device__ __forceinline__ bool flag_wait_bounded(const volatile uint32_t* flag, uint32_t value, uint32_t* err,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (*flag >= value) return true;
  const uint64_t start = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (*flag >= value) return true;
    if (global_timer_ns() - start > limit_ns) {
      raise_error(err, DFLASH2_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// One bulk copy global -> shared (this CTA), completing on `bar` with tx bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// order-preserving 64-bit candidate keys
//   bits 63..48  order-preserving image of the bf16 value (NaN -> 0, -0 -> +0)
//   bits 47..16  ~id   (lower id => larger key)
//   bits 15..0   the original bf16 bits (returned as the value)
// A larger key ranks first; key 0 is "empty" and below every real entry.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bf16_order(uint32_t bits) {
  bits &= 0xFFFFu;
  if ((bits & 0x7FFFu) > 0x7F80u) return 0u;   // NaN ranks below -inf
  if (bits == 0x8000u) bits = 0u;              // -0 == +0
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

__device__ __forceinline__ uint64_t make_key(uint32_t bf16_bits, uint32_t id) {
  return (static_cast<uint64_t>(bf16_order(bf16_bits)) << 48) |
         (static_cast<uint64_t>(~id) << 16) | static_cast<uint64_t>(bf16_bits & 0xFFFFu);
}

__device__ __forceinline__ int32_t key_id(uint64_t key) {
  return static_cast<int32_t>(~static_cast<uint32_t>(key >> 16));
}

__device__ __forceinline__ float key_value(uint64_t key) {
  return __uint_as_float(static_cast<uint32_t>(key & 0xFFFFu) << 16);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits) { return __uint_as_float(bits << 16); }

// Order-preserving image of an fp32 score: NaN -> 0 (below -inf), -0 == +0.
__device__ __forceinline__ uint32_t score_order(float v) {
  if (v != v) return 0u;
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// warp-level top-16 over 64-bit keys (one key per lane)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t kmax(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t kmin(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Sorts the warp's 32 keys in descending order (lane 0 = largest): bitonic network.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, x, j);
      const bool desc_block = (lane & k) == 0;
      const bool lower = (lane & j) == 0;
      x = (lower == desc_block) ? kmax(x, o) : kmin(x, o);
    }
  }
  return x;
}

// `top` holds a descending list in lanes 0..15 (lanes 16..31 hold 0); `x` is an
// arbitrary key per lane.  Returns the descending top-16 of the union in lanes
// 0..15 (0 in lanes 16..31).
__device__ __forceinline__ uint64_t warp_merge_top16(uint64_t top, uint64_t x, int lane) {
  x = warp_sort_desc(x, lane);
  // top (desc, 32 long) against x reversed: the elementwise max is bitonic and
  // holds the 32 largest of the union.
  const uint64_t xr = __shfl_sync(0xFFFFFFFFu, x, 31 - lane);
  uint64_t c = kmax(top, xr);
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, c, j);
    c = ((lane & j) == 0) ? kmax(c, o) : kmin(c, o);
  }
  return lane < 16 ? c : 0ull;
}

}  // namespace dflash2
