// Bins over a range of score keys (sm_103a device code).
#pragma once

#include <cstdint>

namespace dsa {

// A monotone map of score keys onto NB bins spread over [lo, hi]:
// bin(k) = floor((k - lo) scale / 2^32) with scale a little below
// 2^32 NB / (hi - lo + 1), so that every bin of the range is used and
// bin(hi) < NB; keys above hi fall in the top bin.  Only monotonicity matters
// to the callers, so the scale is taken from a float quotient rounded down.
template <int NB>
struct BinMap {
  uint32_t lo, scale;
  __device__ __forceinline__ BinMap(uint32_t lo_, uint32_t hi) : lo(lo_) {
    const float q = __fdividef((float)NB * 4294967296.0f, (float)(hi - lo) + 1.0f);
    scale = __float2uint_rz(q * 0.99999f);   // saturates at 2^32 - 1
  }
  __device__ __forceinline__ int operator()(uint32_t k) const {
    return (int)min(__umulhi(k - lo, scale), (uint32_t)NB - 1u);
  }
  // The smallest key of bin b: lo + ceil(b 2^32 / scale).
  __device__ __forceinline__ uint32_t bottom(int b) const {
    const uint64_t d = (((uint64_t)b << 32) + scale - 1u) / scale;
    const uint64_t k = (uint64_t)lo + d;
    return k > 0xffffffffull ? 0xffffffffu : (uint32_t)k;
  }
};

}  // namespace dsa
