// Division of non-negative 32-bit integers by a divisor fixed at launch time.
//
// The interleaved sharding maps token ids with divisions by I, I*S, S and the
// block size, all known on the host.  A GPU has no integer divider, so each
// such division is replaced by a multiply-high and a shift with a magic
// number computed once on the host: the round-up method of T. Granlund and
// P. L. Montgomery, "Division by Invariant Integers using Multiplication"
// (PLDI 1994), section 4.  With l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, for 0 <= n < 2^31:
//     n / d = (mulhi(m, n) + n) >> l
// (mulhi(m, n) < n, so the sum cannot overflow 32 bits for n < 2^31).
//
// Plain C++ so that a host-only test can check it exhaustively; the device
// path uses the __umulhi intrinsic.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DSA_HD __host__ __device__ __forceinline__
#else
#define DSA_HD inline
#endif

namespace dsa {

struct FastDiv {
  uint32_t d;  // divisor (>= 1)
  uint32_t m;  // magic multiplier
  uint32_t l;  // shift

  FastDiv() : d(1), m(1), l(0) {}
  explicit FastDiv(uint32_t divisor) : d(divisor ? divisor : 1) {
    l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  }
};

DSA_HD uint32_t mulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __umulhi(a, b);
#else
  return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}

// n / f.d for 0 <= n < 2^31.
DSA_HD uint32_t fdiv(uint32_t n, const FastDiv& f) { return (mulhi32(f.m, n) + n) >> f.l; }

// n / f.d and n % f.d together.
DSA_HD uint32_t fdivmod(uint32_t n, const FastDiv& f, uint32_t* rem) {
  const uint32_t q = fdiv(n, f);
  *rem = n - q * f.d;
  return q;
}

}  // namespace dsa
