// Rotation signs of the random Hadamard transform, shared by host and device code
// of the library.  s_i = -1 when bit 63 of SplitMix64's first output from state
// seed + (layer << 32 | head << 16 | i) is set.  SplitMix64 is the generator of
// Steele, Lea & Flood (2014): add the golden-ratio increment, then two
// xor-shift-multiply rounds and a final xor-shift.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define TQ_HD __host__ __device__ __forceinline__
#else
#define TQ_HD inline
#endif

namespace tq {

TQ_HD uint64_t splitmix64_first(uint64_t state) {
  uint64_t z = state + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

TQ_HD bool sign_negative(uint64_t seed, int layer, int head, int i) {
  const uint64_t ctr = (static_cast<uint64_t>(static_cast<uint32_t>(layer)) << 32) |
                       (static_cast<uint64_t>(static_cast<uint32_t>(head)) << 16) | static_cast<uint32_t>(i);
  return (splitmix64_first(seed + ctr) >> 63) != 0;
}

}  // namespace tq
