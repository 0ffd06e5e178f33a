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

// Digits, most significant first: bits [31:21], [20:10], [9:0].
__host__ __device__ constexpr int digit_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__host__ __device__ constexpr int digit_bins(int pass) { return pass == 2 ? 1024 : 2048; }

// After sm.hist holds the NB-bin histogram of a digit: find the bin holding
// the need-th key counted from the top; sm.bin / sm.above / sm.count get the
// bin, the keys in higher bins and the keys in the bin.  Ends with a barrier.
template <int NT, int NB>
__device__ __forceinline__ void find_bin(int need, SelectSmem& sm) {
  constexpr int per = NB / NT;
  static_assert(per >= 1 && NB % NT == 0, "bins per thread");
  const int tid = threadIdx.x;
  int c[per];
  int local = 0;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    c[j] = (int)sm.hist[NB - 1 - (tid * per + j)];
    local += c[j];
  }
  int total;
  int running = block_exclusive_scan(local, sm.scan, &total);
#pragma unroll
  for (int j = 0; j < per; ++j) {
    if (running < need && running + c[j] >= need) {
      sm.bin = NB - 1 - (tid * per + j);
      sm.above = running;
      sm.count = c[j];
    }
    running += c[j];
  }
  __syncthreads();
}

// Radix select resumed at digit `pass0` with the digits above already fixed:
// only keys k with (k & mask) == prefix take part, and `need` counts from the
// top of that group.  visit(f) must call f(k) once for every key the calling
// thread holds (keys outside the group are filtered here).  Requires
// 1 <= need < (keys in the group).  Stops early when the bin holding the
// need-th key is taken whole (take_eq = 0).  *eq gets the size of the last
// bin (at full resolution: the number of keys equal to thr).  NT threads in
// {256, 512, 1024}; every thread calls it; ends with a barrier.
template <int NT, typename Visit>
__device__ SelectResult radix_select_from(int pass0, uint32_t prefix, uint32_t mask, int need,
                                          Visit visit, SelectSmem& sm, int* eq) {
  static_assert(NT == 256 || NT == 512 || NT == 1024, "block size");
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int pass = pass0; pass < 3; ++pass) {
    const int shift = digit_shift(pass);
    const int nb = digit_bins(pass);
    for (int b = tid; b < nb; b += NT) sm.hist[b] = 0u;
    __syncthreads();
    visit([&](uint32_t k) {
      if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & (nb - 1)], 1u);
    });
    __syncthreads();
    if (nb == 2048) find_bin<NT, 2048>(need, sm);
    else find_bin<NT, 1024>(need, sm);
    const int b = sm.bin, above = sm.above, count = sm.count;
    need -= above;
    prefix |= (uint32_t)b << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    *eq = count;
    __syncthreads();
    if (count == need) return SelectResult{prefix - 1u, 0};  // the whole bin is in
  }
  return SelectResult{prefix, need};
}

// The need-th largest of all threads' keys (visit as above).
template <int NT, typename Visit>
__device__ SelectResult radix_select_visit(int need, Visit visit, SelectSmem& sm) {
  int eq;
  return radix_select_from<NT>(0, 0u, 0u, need, visit, sm, &eq);
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
