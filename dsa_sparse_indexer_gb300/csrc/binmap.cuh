// Bins linear in the score over a range (sm_103a device code).
#pragma once

#include <cstdint>

namespace dsa {

// NB bins linear in the score between fmin and fmax: the bin of f is the low
// log2(NB) bits of v = fma(f, scale, c), where c puts fmin at 2^23 + 1 and
// scale = (NB - 3) / (fmax - fmin) keeps fmax below 2^23 + NB - 1.  Every
// float in [2^23, 2^24) is an integer, so the FFMA's rounding replaces a
// float-to-int conversion.  A rounded product and sum never reverse two
// scores, so bins are monotone in the score; callers check once that v(fmin)
// and v(fmax) lie in [2^23, 2^23 + NB), which bounds every score in between.
template <int NB>
struct LinearBinsN {
  float scale, c;
  __device__ __forceinline__ float v(float f) const { return __fmaf_rn(f, scale, c); }
  __device__ __forceinline__ int operator()(float f) const {
    return (int)(__float_as_uint(v(f)) & (uint32_t)(NB - 1));
  }
};

}  // namespace dsa
