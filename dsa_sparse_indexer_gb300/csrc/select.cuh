// Block-wide radix select on 32-bit keys (sm_103a).
#pragma once

#include "common.cuh"

namespace dsa {

// Histogram scratch for one select: 2048 bins plus scan space.
struct SelectSmem {
  uint32_t hist[2048];
  int scan[64];
  int bin, above, count;
};

// Result of a select: an element is among the `need` largest when
//   key > thr,  or  key == thr and it is one of the first `take_eq` elements
//   with key == thr in the caller's tie order.
struct SelectResult {
  uint32_t thr;
  int take_eq;
};

// Finds the `need`-th largest key among all threads' keys.  visit(f) must call
// f(k) once for every key the calling thread holds.  Requires
// 1 <= need < (number of keys).  Digits of 11, 11 and 10 bits, most
// significant first; stops early when the bin holding the need-th key is
// taken whole.  NT threads, NT in {256, 512, 1024}; every thread must call it.
template <int NT, typename Visit>
__device__ SelectResult radix_select_visit(int need, Visit visit, SelectSmem& sm) {
  static_assert(NT == 256 || NT == 512 || NT == 1024, "block size");
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int b = tid; b < nb; b += NT) sm.hist[b] = 0u;
    __syncthreads();
    visit([&](uint32_t k) {
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & (nb - 1)], 1u);
    });
    __syncthreads();
    // Thread t owns bins nb-1-t*per ... (highest first); scan counts from the top.
    const int per = nb / NT;
    int local = 0;
    for (int j = 0; j < per; ++j) local += (int)sm.hist[nb - 1 - (tid * per + j)];
    int total;
    int running = block_exclusive_scan(local, sm.scan, &total);
    for (int j = 0; j < per; ++j) {
      const int b = nb - 1 - (tid * per + j);
      const int c = (int)sm.hist[b];
      if (running < need && running + c >= need) {
        sm.bin = b;
        sm.above = running;
        sm.count = c;
      }
      running += c;
    }
    __syncthreads();
    const int b = sm.bin, above = sm.above, count = sm.count;
    need -= above;
    prefix |= (uint32_t)b << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    __syncthreads();
    if (count == need) return SelectResult{prefix - 1u, 0};  // the whole bin is in
  }
  return SelectResult{prefix, need};
}

// The same over elements i in [0, n), strided over the block; key_at(i, &k)
// returns whether element i takes part.
template <int NT, typename KeyAt>
__device__ SelectResult radix_select(int n, int need, KeyAt key_at, SelectSmem& sm) {
  auto visit = [&](auto&& f) {
    for (int i = threadIdx.x; i < n; i += NT) {
      uint32_t k;
      if (key_at(i, k)) f(k);
    }
  };
  return radix_select_visit<NT>(need, visit, sm);
}

}  // namespace dsa
