// Host-only check of the library's invariant-divisor division (fastdiv.h):
// every divisor 1..70000 against many dividends, plus the extremes, below 2^31.
#include <stdint.h>
#include <stdio.h>

#include "fastdiv.h"

int main() {
  uint64_t checked = 0, state = 0x9E3779B97F4A7C15ull;
  for (uint32_t d = 1; d <= 70000; ++d) {
    const dsa::FastDiv f(d);
    uint32_t probes[64];
    int np = 0;
    const uint32_t fixed[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 2 * d,
                              0x7fffffffu, 0x7ffffffeu, 0x7fffffffu - (0x7fffffffu % d)};
    for (uint32_t v : fixed) probes[np++] = v & 0x7fffffffu;
    while (np < 64) {
      state ^= state << 13; state ^= state >> 7; state ^= state << 17;
      probes[np++] = (uint32_t)(state & 0x7fffffffu);
    }
    for (int i = 0; i < np; ++i) {
      const uint32_t n = probes[i];
      uint32_t r;
      const uint32_t q = dsa::fdivmod(n, f, &r);
      if (q != n / d || r != n % d) {
        printf("FAIL d=%u n=%u q=%u r=%u\n", d, n, q, r);
        return 1;
      }
      ++checked;
    }
  }
  // every dividend for a few divisors the sharding uses
  const uint32_t ds[] = {1, 2, 3, 4, 5, 7, 8, 16, 32, 35, 64, 128};
  for (uint32_t d : ds) {
    const dsa::FastDiv f(d);
    for (uint32_t n = 0; n < (1u << 22); ++n) {
      if (dsa::fdiv(n, f) != n / d) {
        printf("FAIL d=%u n=%u\n", d, n);
        return 1;
      }
      ++checked;
    }
  }
  printf("ok %llu\n", (unsigned long long)checked);
  return 0;
}
