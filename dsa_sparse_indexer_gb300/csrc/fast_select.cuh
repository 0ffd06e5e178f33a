// The K-th largest of register-resident score keys, exactly, without a radix
// pass over all keys (sm_103a).
//
// Each of the NT threads holds V float4 rows of keys, key[j][c] at a slot
// given by the caller (slots order ties: the smaller slot ranks first); key 0
// marks an empty slot.  Steps:
//   1. a 256-bin histogram of one key per float4 row per thread (V samples),
//      linear in the score over the samples' range, proposes a floor a little
//      below the K-th key (about 1.15 K keys at or above it); when the
//      selected sample bin is crowded (an outlier stretching the range) a
//      second 256-bin histogram inside it, linear in the key, refines it;
//   2. a 2048-bin histogram of the keys at or above the floor, spread over
//      [floor, max key], locates the bin b* holding the K-th key;
//   3. the members of b* (at most kFsRankCap) are ranked on (key, ~slot); the
//      one with K - 1 - (keys above b*) keys above it is the threshold.
// Bins other than b* may be crowded; only b* is ranked.  Returns false when
// the floor misses (fewer than K keys at or above it) or b* is crowded: the
// caller then falls back to a radix select.
#pragma once

#include "common.cuh"
#include "reg_topk.cuh"

namespace dsa {

constexpr int kFsBins = 2048;
constexpr int kFsSampleBins = 256;
constexpr int kFsRankCap = 256;

struct FastSelectSmem {
  uint32_t bins[kFsBins];
  uint32_t scnt[kFsSampleBins];
  // Stores are 32-bit: 64-bit stores of (key, slot) pairs made the compiler
  // move the callers' register keys to local memory.
  uint32_t bst_k[kFsRankCap];   // members of b*: score key
  uint32_t bst_s[kFsRankCap];   // and slot
  int scan[33];
  int nsv, nb, bstar, above, bcnt, scount, sabove, sbin, gt, eq;
  uint32_t smin, smax, kmin, kmax, sfloor;
  unsigned long long thr64;
};

// Outcome: a slot wins iff key > thr or (key == thr and slot <= last); with
// kCounts, gt keys are above thr and eq keys equal it (K - gt of the ties win).
struct FastSelectResult {
  uint32_t thr, last;
  int gt, eq;
};

// n: the number of nonzero keys (n > K).  kmn / kmx: this thread's smallest
// nonzero and largest key.  Every thread calls it.  On true it ends with a
// barrier; on false the caller must synchronise before reusing `sm`.
template <int NT, int V, bool kCounts = false, typename SlotOf>
__device__ bool fast_select(const uint32_t (&key)[V][4], int n, int K, uint32_t kmn,
                            uint32_t kmx, SlotOf slot_of, FastSelectSmem& sm,
                            FastSelectResult* out) {
  static_assert(V >= 4, "one sample per float4 row, four rows");
  using ull = unsigned long long;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int b = tid; b < kFsSampleBins; b += NT) sm.scnt[b] = 0u;
  for (int b = tid; b < kFsBins; b += NT) sm.bins[b] = 0u;
  if (tid == 0) {
    sm.nsv = 0;
    sm.nb = 0;
    sm.smin = 0xffffffffu;
    sm.smax = 0u;
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
  }
  // Samples: one lane of each of four spread float4 rows.
  auto sample = [&](int i) { return key[(i * V) / 4][i]; };
  {
    int ns = 0;
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k = sample(i);
      ns += k != 0u;
      mx = max(mx, k);
      mn = min(mn, k ? k : 0xffffffffu);
    }
    ns = __reduce_add_sync(kFull, ns);
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    kmn = __reduce_min_sync(kFull, kmn);
    kmx = __reduce_max_sync(kFull, kmx);
    __syncthreads();
    if (lane == 0) {
      atomicMin(&sm.kmin, kmn);
      atomicMax(&sm.kmax, kmx);
      if (ns) {
        atomicAdd(&sm.nsv, ns);
        atomicMin(&sm.smin, mn);
        atomicMax(&sm.smax, mx);
      }
    }
  }
  __syncthreads();
  uint32_t floor = sm.kmin;   // without a sample floor: every key
  const uint32_t kmax = sm.kmax;
  const int nsv = sm.nsv;
  if (n * 4 > K * 5 && nsv >= 64) {
    const uint32_t smin = sm.smin, smax = sm.smax;
    // Bins linear in the score: bin(k) = (score(k) - fmin) * fscale, clamped.
    const float fmin = key_score(smin), fspan = key_score(smax) - fmin;
    const float fscale = fspan > 0.f ? (float)kFsSampleBins / fspan : 0.f;
    auto sbin = [&](uint32_t k) {
      return min(kFsSampleBins - 1, max(0, (int)((key_score(k) - fmin) * fscale)));
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k = sample(i);
      if (k) atomicAdd(&sm.scnt[sbin(k)], 1u);
    }
    __syncthreads();
    // Expected samples among the winners: nsv * K / n; take 1/8 more and 16.
    const int target = min(nsv, (int)((float)nsv * (float)K * 1.125f / (float)n) + 16);
    const int local = tid < kFsSampleBins ? (int)sm.scnt[kFsSampleBins - 1 - tid] : 0;
    int tot;
    const int run = block_exclusive_scan(local, sm.scan, &tot);
    if (tid < kFsSampleBins && run < target && run + local >= target) {
      sm.sbin = kFsSampleBins - 1 - tid;
      sm.scount = local;
      sm.sabove = run;
      sm.sfloor = 0xffffffffu;
    }
    __syncthreads();
    // The floor: the smallest sample in the selected bin (so every sample of
    // the bin, and the target-th from the top, is at or above it).
    const int selbin = sm.sbin;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k = sample(i);
      if (k && sbin(k) == selbin) atomicMin(&sm.sfloor, k);
    }
    __syncthreads();
    floor = sm.sfloor;
    if (sm.scount > 32) {
      // Crowded bin: refine inside [floor, largest sample of the bin], linear in the key.
      const uint32_t top = fscale > 0.f ? score_key(fmin + (float)(selbin + 1) / fscale) : smax;
      const int ssh2 = max(0, (32 - __clz((int)(max(top, floor) - floor))) - 8);
      const int target2 = target - sm.sabove;
      for (int b = tid; b < kFsSampleBins; b += NT) sm.scnt[b] = 0u;
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t k = sample(i);
        if (k && sbin(k) == selbin)
          atomicAdd(&sm.scnt[min(kFsSampleBins - 1, (int)((k - floor) >> ssh2))], 1u);
      }
      __syncthreads();
      const int local2 = tid < kFsSampleBins ? (int)sm.scnt[kFsSampleBins - 1 - tid] : 0;
      const int run2 = block_exclusive_scan(local2, sm.scan, &tot);
      if (tid < kFsSampleBins && run2 < target2 && run2 + local2 >= target2)
        sm.sfloor = floor + ((uint32_t)(kFsSampleBins - 1 - tid) << ssh2);
      __syncthreads();
      floor = sm.sfloor;
    }
  }

  // Histogram of the keys >= floor over [floor, kmax].
  const int sh2 = max(0, (32 - __clz((int)(kmax - floor))) - 11);   // range >> sh2 < 2048
  auto bin_of = [&](uint32_t k) { return (int)((k - floor) >> sh2); };
#pragma unroll
  for (int j = 0; j < V; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (key[j][c] >= floor && key[j][c]) atomicAdd(&sm.bins[bin_of(key[j][c])], 1u);
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
      bm |= (uint32_t)(k >= floor && k && bin_of(k) == bstar) << (4 * j + c);
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
