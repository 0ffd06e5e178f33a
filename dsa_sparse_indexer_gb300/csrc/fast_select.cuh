// The K-th largest of a CTA's scores, exactly, without a radix pass over all
// of them (sm_103a).
//
// Each of the NT threads owns V float4 rows of scores, read through get4h(j)
// for the histogram and get4(j) afterwards (registers or shared memory),
// element c of row j at a slot given by the caller (slots order ties: the smaller slot ranks first); -inf
// marks an empty slot (the fast path runs only when every real score is
// finite).  Steps:
//   1. a 2048-bin histogram of every score, the bins linear in the score
//      between the smallest and the largest, locates the bin b* holding the
//      K-th score (a normal-like row leaves a few dozen scores there);
//   2. the members of b* (at most kFsRankCap) are ranked on (score key, ~slot);
//      the one with K - 1 - (scores above b*) members above it is the
//      threshold.
// Bins other than b* may be crowded; only b* is ranked.  Returns false when a
// score is infinite, the range is empty or too narrow for the bin map, b* is
// the lowest bin or crowded (an outlier stretching the range, heavy ties):
// the caller then falls back to a radix select.
//
// The bin of a score f is read off the bits of v = fma(f, scale, c), where c
// puts the smallest score at 2^23 + 1 and scale = 2045 / range keeps the
// largest below 2^23 + 2047: every float in [2^23, 2^24) is an integer, so the
// FFMA's rounding replaces a float-to-int conversion and the low 11 bits of v
// are the bin (the exponent field of 2^23 has none set).  A rounded product
// and sum never reverse two scores, so bins are monotone in the score; the
// two ends are checked once, which bounds every score in between.  An empty
// slot (-inf) gives v = -inf, whose low 11 bits are 0: it only adds to bin 0,
// which is never b* on this path.
#pragma once

#include "common.cuh"
#include "reg_topk.cuh"

namespace dsa {

constexpr int kFsBins = 2048;
constexpr int kFsRankCap = 256;

struct alignas(16) FastSelectSmem {
  uint32_t bins[kFsBins];
  // Stores are 32-bit: 64-bit stores of (key, slot) pairs made the compiler
  // move the callers' register scores to local memory.
  uint32_t bst_k[kFsRankCap];   // members of b*: score key
  uint32_t bst_s[kFsRankCap];   // and slot
  int scan[33];
  int nb, bstar, above, bcnt, eq;
  uint32_t wmin[32], wmax[32];   // each warp's smallest and largest score key
  unsigned long long thr64;
};

// Outcome: a slot wins iff f > thr or (f == thr and slot <= last); eq scores
// equal thr (eq == 1: the threshold's own, so every f >= thr wins).
struct FastSelectResult {
  float thr;
  uint32_t last;
  int eq;
};

// The bin of a score: the low 11 bits of fma(f, scale, c) (see above).
struct LinearBins {
  float scale, c;
  __device__ __forceinline__ float v(float f) const { return __fmaf_rn(f, scale, c); }
  __device__ __forceinline__ int operator()(float f) const {
    return (int)(__float_as_uint(v(f)) & (uint32_t)(kFsBins - 1));
  }
};

// f4at: element c of a float4.  fast_select: more than K real scores; fmn / fmx
// this thread's smallest and largest real score (+inf / -inf if none); every
// thread calls it; true ends with a barrier, false needs one before sm is reused.
__device__ __forceinline__ float f4at(const float4& v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}

template <int NT, int V, typename Get4H, typename Get4, typename SlotOf, typename ScoreAt>
__device__ bool fast_select(Get4H get4h, Get4 get4, int K, float fmn, float fmx, SlotOf slot_of,
                            ScoreAt score_at, FastSelectSmem& sm, FastSelectResult* out) {
  using ull = unsigned long long;
  constexpr int W = NT / 32;
  static_assert(W <= 32, "one lane per warp in the reductions");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int b = tid; b < kFsBins; b += NT) sm.bins[b] = 0u;
  if (tid == 0) sm.nb = 0;
  {
    const uint32_t mn = __reduce_min_sync(kFull, score_key(fmn));
    const uint32_t mx = __reduce_max_sync(kFull, score_key(fmx));
    if (lane == 0) {
      sm.wmin[warp] = mn;
      sm.wmax[warp] = mx;
    }
  }
  __syncthreads();
  // Every warp reduces the warps' keys itself (no second barrier).
  const uint32_t kmin = __reduce_min_sync(kFull, lane < W ? sm.wmin[lane] : 0xffffffffu);
  const uint32_t kmax = __reduce_max_sync(kFull, lane < W ? sm.wmax[lane] : 0u);
  const float fmin = key_score(kmin), fmax = key_score(kmax);
  constexpr float kTwo23 = 8388608.0f;
  const float scale = __fdividef(2045.0f, fmax - fmin);
  const LinearBins bin_of{scale, (kTwo23 + 1.0f) - fmin * scale};
  // Same values in every thread: all of them return here or none.
  if (!(fmax > fmin) || !isfinite(fmin) || !isfinite(fmax) || !isfinite(scale) ||
      !(bin_of.v(fmin) >= kTwo23) || !(bin_of.v(fmax) <= kTwo23 + (float)(kFsBins - 1)))
    return false;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float4 v = get4h(j);
#pragma unroll
    for (int c = 0; c < 4; ++c) atomicAdd(&sm.bins[bin_of(f4at(v, c))], 1u);
  }
  __syncthreads();
  {
    constexpr int per = kFsBins / NT;
    static_assert(per % 2 == 0, "bins read in pairs");
    const int g = kFsBins - per * (tid + 1);
    int local = 0;
#pragma unroll
    for (int j = 0; j < per; j += 2) {
      const uint2 c = *reinterpret_cast<const uint2*>(&sm.bins[g + j]);
      local += (int)(c.x + c.y);
    }
    // Exclusive prefix over the block with one barrier: a warp scan, the
    // warps' totals, and every warp adding up the totals of the warps before.
    const int incl = warp_inclusive_scan(local);
    if (lane == 31) sm.scan[warp] = incl;
    __syncthreads();
    const int ws = lane < W ? sm.scan[lane] : 0;
    const int wincl = warp_inclusive_scan(ws);
    int run = __shfl_sync(kFull, wincl - ws, warp) + incl - local;
    // One thread's bins hold the K-th position: it finds b* among them (the
    // counts read again rather than held in registers beside the scores).
    if (run < K && run + local >= K) {
      for (int j = 0; j < per; ++j) {
        const int b = g + per - 1 - j, c = (int)sm.bins[b];
        if (run + c >= K) {
          sm.bstar = b;
          sm.above = run;
          sm.bcnt = c;
          break;
        }
        run += c;
      }
    }
  }
  __syncthreads();
  // Bin 0 also counts the empty slots: the K-th score must lie above it.
  if (sm.bstar == 0 || sm.bcnt > kFsRankCap) return false;

  // Members of b* (v is an integer-valued float: the bin test is one compare),
  // then the exact threshold by ranking them.
  const int bcnt = sm.bcnt, take = K - sm.above;
  const float vstar = kTwo23 + (float)sm.bstar;
  uint32_t bm = 0u;   // bit 4 j + c: slot (j, c) is in b*
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float4 v = get4(j);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      bm |= (uint32_t)(bin_of.v(f4at(v, c)) == vstar) << (4 * j + c);
  }
  if (__any_sync(kFull, bm != 0u)) {   // most warps hold no member
    const int mine = __popc(bm);
    const int incl = warp_inclusive_scan(mine);
    int b0 = 0;
    if (lane == 31) b0 = atomicAdd(&sm.nb, incl);
    int q = __shfl_sync(kFull, b0, 31) + incl - mine;
    // Most lanes hold no member: walk the set bits, each member's score read
    // back by its slot (the value loaded into f; a register array cannot be
    // indexed by a run-time bit).
    while (bm != 0u) {
      const int k = __ffs((int)bm) - 1;
      bm &= bm - 1u;
      const uint32_t sl = slot_of(k >> 2, k & 3);
      sm.bst_k[q] = score_key(score_at(sl));
      sm.bst_s[q] = sl;
      ++q;
    }
  }
  __syncthreads();
  // Rank on (score key, ~slot): the member with take - 1 above it.  It also
  // counts the members with its score.
  auto member = [&](int i) { return ((ull)sm.bst_k[i] << 32) | ~sm.bst_s[i]; };
  for (int i = tid; i < bcnt; i += NT) {
    const ull x = member(i);
    const uint32_t xk = (uint32_t)(x >> 32);
    int gt = 0, eq = 0;
    for (int q = 0; q < bcnt; ++q) {
      gt += member(q) > x;
      eq += sm.bst_k[q] == xk;
    }
    if (gt == take - 1) {
      sm.thr64 = x;
      sm.eq = eq;
    }
  }
  __syncthreads();
  const ull thr64 = sm.thr64;
  out->thr = key_score((uint32_t)(thr64 >> 32));
  out->last = ~(uint32_t)thr64;
  out->eq = sm.eq;
  return true;
}

}  // namespace dsa
