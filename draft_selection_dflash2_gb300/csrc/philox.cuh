// philox.cuh -- Philox4x32-10 counter-based generator (Salmon, Moraes, Dror and
// Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11), device side.
//
// Stream layout used by the library: counter = (b, t | stream << 24, offset_lo,
// offset_hi), key = (seed_lo, seed_hi); a uniform is (x0 >> 8) * 2^-24.
// Streams: 0 = walk draw, 1 = verification accept test, 2 = residual / bonus draw.
#pragma once

#include <stdint.h>

namespace dflash2 {

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t out[4]) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// The 24 random bits of (b, t, stream, offset) under key seed: x0 >> 8.
__device__ __forceinline__ uint32_t philox_bits24(uint64_t seed, uint32_t b, uint32_t t, uint32_t stream,
                                                  uint64_t offset) {
  uint32_t out[4];
  philox4x32_10(b, t | (stream << 24), static_cast<uint32_t>(offset),
                static_cast<uint32_t>(offset >> 32), static_cast<uint32_t>(seed),
                static_cast<uint32_t>(seed >> 32), out);
  return out[0] >> 8;
}

// Uniform in [0, 1) with 24 random bits, as a double (exact).
__device__ __forceinline__ double philox_uniform24(uint64_t seed, uint32_t b, uint32_t t,
                                                   uint32_t stream, uint64_t offset) {
  return static_cast<double>(philox_bits24(seed, b, t, stream, offset)) * (1.0 / 16777216.0);
}

}  // namespace dflash2
