// The K-th largest of register-resident score keys, exactly, without a radix
// pass over all keys (sm_103a).
//
// Each of the NT threads holds V float4 rows of keys, key[j][c] at a slot
// given by the caller (slots order ties: the smaller slot ranks first); key 0
// marks an empty slot.  Steps:
//   1. a 2048-bin histogram of every key, the bins linear in the score between
//      the smallest and the largest key, locates the bin b* holding the K-th
//      key (a normal-like row leaves a few dozen keys there);
//   2. the members of b* (at most kFsRankCap) are ranked on (key, ~slot); the
//      one with K - 1 - (keys above b*) keys above it is the threshold.
// Bins other than b* may be crowded; only b* is ranked.  Returns false when a
// score is infinite, the range is empty or b* is crowded (an outlier
// stretching the range, heavy ties): the caller then falls back to a radix
// select.
#pragma once

#include "common.cuh"
#include "reg_topk.cuh"

namespace dsa {

constexpr int kFsBins = 2048;
constexpr int kFsRankCap = 256;

struct FastSelectSmem {
  uint32_t bins[kFsBins];
  // Stores are 32-bit: 64-bit stores of (key, slot) pairs made the compiler
  // move the callers' register keys to local memory.
  uint32_t bst_k[kFsRankCap];   // members of b*: score key
  uint32_t bst_s[kFsRankCap];   // and slot
  int scan[33];
  int nb, bstar, above, bcnt, gt, eq;
  uint32_t kmin, kmax;
  unsigned long long thr64;
};

// Outcome: a slot wins iff key > thr or (key == thr and slot <= last); with
// kCounts, gt keys are above thr and eq keys equal it (K - gt of the ties win).
struct FastSelectResult {
  uint32_t thr, last;
  int gt, eq;
};

// More than K nonzero keys.  kmn / kmx: this thread's smallest nonzero and
// largest key.  Every thread calls it.  On true it ends with a barrier; on
// false the caller must synchronise before reusing `sm`.
template <int NT, int V, bool kCounts = false, typename SlotOf>
__device__ bool fast_select(const uint32_t (&key)[V][4], int K, uint32_t kmn, uint32_t kmx,
                            SlotOf slot_of, FastSelectSmem& sm, FastSelectResult* out) {
  using ull = unsigned long long;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int b = tid; b < kFsBins; b += NT) sm.bins[b] = 0u;
  if (tid == 0) {
    sm.nb = 0;
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
  }
  {
    const uint32_t mn = __reduce_min_sync(kFull, kmn), mx = __reduce_max_sync(kFull, kmx);
    __syncthreads();
    if (lane == 0) {
      atomicMin(&sm.kmin, mn);
      atomicMax(&sm.kmax, mx);
    }
  }
  __syncthreads();
  // Bins linear in the score over [smallest, largest key]: a normal-like row
  // leaves a few dozen keys in the bin of the K-th.  Monotone in the key (a
  // rounded difference, a rounded positive product and a truncation never
  // reverse the order of two scores).  Same values in every thread.
  const float fmin = key_score(sm.kmin), fmax = key_score(sm.kmax);
  const float fscale = __fdividef((float)kFsBins, fmax - fmin);
  if (!(fmax > fmin) || !isfinite(fmin) || !isfinite(fmax) || !isfinite(fscale)) return false;
  auto bin_of = [&](uint32_t k) {
    return min(kFsBins - 1, (int)__float2uint_rz((key_score(k) - fmin) * fscale));
  };
#pragma unroll
  for (int j = 0; j < V; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (key[j][c]) atomicAdd(&sm.bins[bin_of(key[j][c])], 1u);
  __syncthreads();
  int total;
  {
    constexpr int per = kFsBins / NT;
    const int g = kFsBins - per * (tid + 1);
    int cnt[per];
    int local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      cnt[j] = (int)sm.bins[g + per - 1 - j];
      local += cnt[j];
    }
    int run = block_exclusive_scan(local, sm.scan, &total);
#pragma unroll
    for (int j = 0; j < per; ++j) {
      if (run < K && run + cnt[j] >= K) {
        sm.bstar = g + per - 1 - j;
        sm.above = run;
        sm.bcnt = cnt[j];
      }
      run += cnt[j];
    }
  }
  __syncthreads();
  if (total < K || sm.bcnt > kFsRankCap) return false;

  // Members of b*, then the exact threshold by ranking them.
  const int bstar = sm.bstar, bcnt = sm.bcnt, take = K - sm.above;
  uint32_t bm = 0u;   // bit 4 j + c: slot (j, c) is in b*
#pragma unroll
  for (int j = 0; j < V; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t k = key[j][c];
      bm |= (uint32_t)(k && bin_of(k) == bstar) << (4 * j + c);
    }
  if (__any_sync(kFull, bm != 0u)) {   // most warps hold no member
    const int mine = __popc(bm);
    const int incl = warp_inclusive_scan(mine);
    int b0 = 0;
    if (lane == 31) b0 = atomicAdd(&sm.nb, incl);
    int q = __shfl_sync(kFull, b0, 31) + incl - mine;
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (bm >> (4 * j + c) & 1u) {
          sm.bst_k[q] = key[j][c];
          sm.bst_s[q] = slot_of(j, c);
          ++q;
        }
  }
  __syncthreads();
  // Rank on (score key, ~slot): the member with take - 1 above it.
  auto member = [&](int i) { return ((ull)sm.bst_k[i] << 32) | ~sm.bst_s[i]; };
  for (int i = tid; i < bcnt; i += NT) {
    const ull x = member(i);
    int gt = 0;
    for (int q = 0; q < bcnt; ++q) gt += member(q) > x;
    if (gt == take - 1) sm.thr64 = x;
  }
  __syncthreads();
  const ull thr64 = sm.thr64;
  const uint32_t thr = (uint32_t)(thr64 >> 32);
  out->thr = thr;
  out->last = ~(uint32_t)thr64;
  out->gt = out->eq = -1;
  if (kCounts) {
    if (tid == 0) {
      int gt = 0, eq = 0;
      for (int q = 0; q < bcnt; ++q) {
        gt += sm.bst_k[q] > thr;
        eq += sm.bst_k[q] == thr;
      }
      sm.gt = sm.above + gt;
      sm.eq = eq;
    }
    __syncthreads();
    out->gt = sm.gt;
    out->eq = sm.eq;
  }
  return true;
}

}  // namespace dsa
