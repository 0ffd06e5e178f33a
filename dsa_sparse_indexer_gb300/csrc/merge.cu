// Stable global top-K of the gathered (score, global id) candidates.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 实现拆解 item 1 (`stable_topk_from_gathered_candidates_cutedsl`, a
// radix selector) and section 关键源码片段 (the all_gathered [batch, S*topk, 2]
// buffer; topk_indices overwritten with global ids, -1 for padding).
//
// One CTA per row; every candidate is ranked by its 64-bit key
// (score_key << 32 | ~id), so ties go to the smaller id.  Batches that fit one
// wave (up to 16 candidates per thread) take the latency kernel
// (merge_lin_kernel): every candidate in registers, one histogram linear in
// the score over their range.  Otherwise rows of up to 32 candidates per
// thread (C <= 32768) take the throughput kernel (merge_fast_kernel): a
// sampled floor, a compact list of the candidates above it, bins over the
// list's key range that give the winners' output ranges, and ranking inside
// each (small) bin (both kernels rank the same way).  Larger rows (merge_kernel) are read
// from global memory (L2 after the first pass): a radix select on the score
// key, and, only when the K-th score is tied, a second one on the inverted
// id; the K winners are then put in rank order by a bitonic sort.
#include "binmap.cuh"
#include "checks.h"
#include "common.cuh"
#include "reg_topk.cuh"
#include "select.cuh"

namespace dsa {
namespace {

// Block-wide exclusive prefix sum with one __syncthreads(): every warp scans
// the warp totals itself instead of waiting for one warp to publish them.
// The caller puts a barrier between this call and the next write to
// `scratch` (at least blockDim.x / 32 ints).
__device__ __forceinline__ int block_exclusive_scan_1bar(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  const int w = lane < nwarps ? scratch[lane] : 0;
  int incl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  return __shfl_sync(kFull, incl - w, warp) + x - v;
}

constexpr int kMergeThreads = 1024;
constexpr int kMaxK = 2048;

struct MergeSmem {
  SelectSmem sel;
  unsigned long long win[kMaxK];
  int nwin;
  int valid_count;
  int tied;
};

__global__ void __launch_bounds__(kMergeThreads, 1)
    merge_kernel(const float* __restrict__ cand, int C, int K, int32_t* __restrict__ ids,
                 float* __restrict__ scores) {
  __shared__ MergeSmem sm;
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = blockIdx.x;
  const float2* data = reinterpret_cast<const float2*>(cand) + (int64_t)r * C;

  if (tid == 0) { sm.nwin = 0; sm.valid_count = 0; sm.tied = 0; }
  __syncthreads();

  // Valid candidates (id >= 0).
  int nv = 0;
  for (int i = tid; i < C; i += kMergeThreads) nv += __float_as_int(data[i].y) >= 0;
  nv = __reduce_add_sync(kFull, nv);
  if (lane == 0) atomicAdd(&sm.valid_count, nv);
  __syncthreads();
  const int valid = sm.valid_count;

  // Winner rule: key32 > thr1, or key32 == thr1 and ~id >= thr2 (when tied).
  uint32_t thr1 = 0;
  bool all = valid <= K, tie = false;
  uint32_t thr2 = 0;
  if (!all) {
    auto key1 = [&](int i, uint32_t& k) {
      const float2 c = data[i];
      k = score_key(c.x);
      return __float_as_int(c.y) >= 0;
    };
    const SelectResult a = radix_select<kMergeThreads>(C, K, key1, sm.sel);
    thr1 = a.thr;
    if (a.take_eq > 0) {
      // Count the tied group; if it is larger than needed, pick the smallest ids.
      int e = 0;
      for (int i = tid; i < C; i += kMergeThreads) {
        const float2 c = data[i];
        e += (__float_as_int(c.y) >= 0 && score_key(c.x) == thr1);
      }
      e = __reduce_add_sync(kFull, e);
      if (lane == 0) atomicAdd(&sm.tied, e);
      __syncthreads();
      const int tied = sm.tied;
      if (tied > a.take_eq) {
        auto key2 = [&](int i, uint32_t& k) {
          const float2 c = data[i];
          const int id = __float_as_int(c.y);
          k = ~(uint32_t)id;
          return id >= 0 && score_key(c.x) == thr1;
        };
        const SelectResult b = radix_select<kMergeThreads>(C, a.take_eq, key2, sm.sel);
        // ids are distinct, so exactly take_eq tied candidates have ~id >= thr2.
        thr2 = b.take_eq > 0 ? b.thr : b.thr + 1u;
        tie = true;
      } else {
        thr1 = thr1 - 1u;  // the whole tied group is in: key32 >= old thr1
      }
    }
  }

  // Gather winners' 64-bit rank keys (order of arrival does not matter).
  for (int base = 0; base < C; base += kMergeThreads) {
    const int i = base + tid;
    bool w = false;
    unsigned long long key = 0ull;
    if (i < C) {
      const float2 c = data[i];
      const int id = __float_as_int(c.y);
      if (id >= 0) {
        const uint32_t k1 = score_key(c.x);
        w = all || k1 > thr1 || (tie && k1 == thr1 && ~(uint32_t)id >= thr2);
        key = ((unsigned long long)k1 << 32) | (unsigned long long)(~(uint32_t)id);
      }
    }
    const unsigned m = __ballot_sync(kFull, w);
    int wbase = 0;
    if (lane == 0 && m) wbase = atomicAdd(&sm.nwin, __popc(m));
    wbase = __shfl_sync(kFull, wbase, 0);
    const int slot = wbase + __popc(m & lanemask_lt());
    if (w && slot < K) sm.win[slot] = key;
  }
  __syncthreads();
  const int nwin = min(sm.nwin, K);
  for (int j = nwin + tid; j < K; j += kMergeThreads) sm.win[j] = 0ull;  // padding sorts last
  __syncthreads();

  // Bitonic sort, descending.
  for (int k = 2; k <= K; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = tid; p < (K >> 1); p += kMergeThreads) {
        const int i = 2 * p - (p & (j - 1));
        const int ixj = i + j;
        const bool desc = (i & k) == 0;
        const unsigned long long a = sm.win[i], b = sm.win[ixj];
        if ((a < b) == desc) { sm.win[i] = b; sm.win[ixj] = a; }
      }
      __syncthreads();
    }
  }

  int32_t* out_ids = ids + (int64_t)r * K;
  float* out_sc = scores ? scores + (int64_t)r * K : nullptr;
  for (int j = tid; j < K; j += kMergeThreads) {
    const unsigned long long key = sm.win[j];
    const bool v = key != 0ull;
    out_ids[j] = v ? (int32_t)(~(uint32_t)(key & 0xffffffffull)) : -1;
    if (out_sc) out_sc[j] = v ? key_score((uint32_t)(key >> 32)) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Throughput path (C <= 32 * NT).  Each thread loads 16 float4 (32
// candidates) in four batches of 4, batch b holding float4 rows
// 4 i + (i + b) mod 4, so every batch spans all shard blocks and all parts of
// each block.  While the second batch is in flight, a histogram of one
// candidate per float4 of the first batch (256 bins linear in the score over
// the samples' range) proposes a floor a little below the K-th score; each
// batch's valid candidates at or above it (about 1.15 K in all) are appended to
// a shared list as raw (score, id) pairs.  If fewer than K made it, or no floor
// could be set (few valid candidates, an infinite sample), every valid
// candidate is listed instead and the list's exact score range is taken.
//
// On the list, a histogram of 2048 bins does two jobs: a scan from the top bin
// finds the bin b* holding the K-th candidate and gives every bin above b* its
// output range, since all of those candidates win.  The bins are spaced
// logarithmically above the floor: the bin of a score f is read off the bit
// pattern of w = f - floor + delta (delta = range / 15), whose top bits count
// 512 bins per octave of w from delta to 16 delta.  A rounded sum and the bit
// pattern of a non-negative float are both monotone, so bins keep the score
// order; and since candidate scores thin out above the floor (the upper tail
// of the shards' winners), bins that widen with the distance from the floor
// hold one or two candidates each, where equal widths hold several near the
// floor.  Winners above b* go into their bin's range as 64-bit rank keys
// (score key << 32 | ~id, so one unsigned compare orders two candidates:
// higher score first, then the smaller id) and are ranked inside it; the
// members of b* are ranked among themselves.  Rows with a crowded bin (heavy
// ties, an outlier stretching the range), a non-finite range or an
// overflowing list take a radix select for the threshold and a bitonic sort.
// Ranked winners are staged in shared memory and written with 16-byte stores.
// ---------------------------------------------------------------------------
using ull = unsigned long long;
constexpr int kMBins = 2048;
constexpr int kSampBins = 256;      // bins of the sample histogram
constexpr int kMListCap = 3072;     // candidates at or above the floor
constexpr int kRankCap = 256;       // most members of b* for the pairwise ranking
constexpr int kFineCap = 64;        // most keys in one bin above b*
constexpr int kQuarter = 4;         // float4 per thread per batch
constexpr int kLogShift = 14;       // 2^(23 - 14) = 512 bins per octave

struct alignas(16) MergeFastSmem {
  union {
    ull l[kMListCap];               // rank keys (latency kernel)
    float2 f[kMListCap];            // raw (score, id) at or above the floor
    ull lb[kMaxK];                  // crowded rows: all winners
    ull out[kMaxK];                 // ranked winners by output position
  } u;
  union {
    // Keys per bin; after the scan the start of the bin's output range
    // (bins are output from the top down), after the scatter its end, which
    // is also the start of the bin below.
    uint32_t end[kMBins];
    SelectSmem sel;                 // crowded rows only
  } h;
  union {
    ull win[kMaxK];                 // winners above b*, by output range
    uint32_t scnt[kSampBins];       // sample histogram (before the list exists)
  } w;
  ull bst[kRankCap];                // members of b*
  int scan[33];
  int nsv, nslots, nlist, nlist2, nb, nwin, bstar, above, bcnt;
  int bmax[2];                      // per level, so that no reset races a read
  uint32_t smin, smax, lmin, lmin2, kmax, kmax2;
  float sfloor;
};

template <int NT>
constexpr int merge_fast_min_blocks() { return NT == 256 ? 4 : (NT == 512 ? 2 : 1); }

__device__ __forceinline__ ull rank_key(float score, float id_bits) {
  const int id = __float_as_int(id_bits);
  return id >= 0 ? ((ull)score_key(score) << 32) | (uint32_t)~id : 0ull;
}

// Rows with crowded bins or an overflowing list.  Among the `count` keys with
// score key >= lo (which hold every winner) the K-th rank key thr64 comes from
// a radix select over score keys, then over ~id of the keys tied at the
// threshold; all winners are then sorted by a bitonic network.  Keys are
// re-read from the row (in L2).
template <int NT>
__device__ __noinline__ void merge_crowded(const float* __restrict__ row, int C, uint32_t lo,
                                           int count, int need, MergeFastSmem& sm,
                                           int32_t* out_ids, float* out_sc) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float2* row2 = reinterpret_cast<const float2*>(row);
  auto rk = [&](int e) {
    const float2 v = __ldg(row2 + e);
    return rank_key(v.x, v.y);
  };
  ull thr64;
  if (count == need) {
    thr64 = (ull)lo << 32;
  } else {
    auto visit = [&](auto&& f) {
      for (int e = tid; e < C; e += NT) {
        const uint32_t k = (uint32_t)(rk(e) >> 32);
        if (k && k >= lo) f(k);
      }
    };
    int eq;
    const SelectResult res = radix_select_from<NT>(0, 0u, 0u, need, visit, sm.h.sel, &eq);
    const uint32_t thr = res.thr;
    if (res.take_eq == 0) {
      thr64 = (ull)(thr + 1u) << 32;
    } else if (res.take_eq == eq) {
      thr64 = (ull)thr << 32;
    } else {
      auto visit_id = [&](auto&& f) {
        for (int e = tid; e < C; e += NT) {
          const ull x = rk(e);
          if ((uint32_t)(x >> 32) == thr) f((uint32_t)x);
        }
      };
      const SelectResult t2 = radix_select_visit<NT>(res.take_eq, visit_id, sm.h.sel);
      thr64 = ((ull)thr << 32) | (t2.take_eq > 0 ? t2.thr : t2.thr + 1u);
    }
  }
  // Gather the winners (warp-aggregated append).
  for (int e0 = 0; e0 < C; e0 += NT) {
    const int e = e0 + tid;
    const ull x = e < C ? rk(e) : 0ull;
    const bool w = x != 0ull && x >= thr64;
    const unsigned bal = __ballot_sync(kFull, w);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(&sm.nwin, __popc(bal));
    base = __shfl_sync(kFull, base, 0);
    const int p = base + __popc(bal & lanemask_lt());
    if (w && p < kMaxK) sm.u.lb[p] = x;
  }
  __syncthreads();
  const int nwin = min(sm.nwin, need);
  int P = 1;
  while (P < nwin) P <<= 1;
  for (int j = nwin + tid; j < P; j += NT) sm.u.lb[j] = 0ull;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int q = tid; q < (P >> 1); q += NT) {
        const int i = 2 * q - (q & (j - 1));
        const bool desc = (i & k) == 0;
        const ull x = sm.u.lb[i], y = sm.u.lb[i + j];
        if ((x < y) == desc) {
          sm.u.lb[i] = y;
          sm.u.lb[i + j] = x;
        }
      }
      __syncthreads();
    }
  }
  for (int q = tid; q < nwin; q += NT) {
    const ull x = sm.u.lb[q];
    out_ids[q] = (int32_t)~(uint32_t)x;
    if (out_sc) out_sc[q] = key_score((uint32_t)(x >> 32));
  }
}

// Entries of a[s0, e) above x.  Bins mostly hold a few keys: the first U
// entries are compared without a loop, so lanes with different bin sizes
// stay together.
template <int U = 4>
__device__ __forceinline__ int count_above(const ull* a, int s0, int e, ull x) {
  int gt = 0;
#pragma unroll
  for (int j = 0; j < U; ++j)
    if (s0 + j < e) gt += a[s0 + j] > x;
  for (int q = s0 + U; q < e; ++q) gt += a[q] > x;
  return gt;
}

// Appends two batches' valid candidates with score >= ffloor to the list as
// raw (score, id) pairs: one pass mask per thread, one warp scan and one
// shared atomic per warp for the positions.  NaN scores fail the comparison.
__device__ __forceinline__ void append_batches(const float4 (&va)[kQuarter],
                                               const float4 (&vb)[kQuarter], float ffloor,
                                               MergeFastSmem& sm, int* counter) {
  const int lane = threadIdx.x & 31;
  uint32_t mask = 0u;   // bit 2 i + h (+ 8 for vb): candidate h of float4 i passes
#pragma unroll
  for (int i = 0; i < kQuarter; ++i) {
    mask |= (uint32_t)(__float_as_int(va[i].y) >= 0 && va[i].x >= ffloor) << (2 * i);
    mask |= (uint32_t)(__float_as_int(va[i].w) >= 0 && va[i].z >= ffloor) << (2 * i + 1);
    mask |= (uint32_t)(__float_as_int(vb[i].y) >= 0 && vb[i].x >= ffloor) << (2 * i + 8);
    mask |= (uint32_t)(__float_as_int(vb[i].w) >= 0 && vb[i].z >= ffloor) << (2 * i + 9);
  }
  const int m = __popc(mask);
  const int incl = warp_inclusive_scan(m);
  int base = 0;
  if (lane == 31 && incl) base = atomicAdd(counter, incl);
  int p = __shfl_sync(kFull, base, 31) + incl - m;
  auto put = [&](const float4& v, int bit) {
    if ((mask >> bit & 1u) && p < kMListCap) sm.u.f[p] = make_float2(v.x, v.y);
    p += mask >> bit & 1u;
    if ((mask >> (bit + 1) & 1u) && p < kMListCap) sm.u.f[p] = make_float2(v.z, v.w);
    p += mask >> (bit + 1) & 1u;
  };
#pragma unroll
  for (int i = 0; i < kQuarter; ++i) put(va[i], 2 * i);
#pragma unroll
  for (int i = 0; i < kQuarter; ++i) put(vb[i], 2 * i + 8);
}

// Log-spaced bins of scores at or above lo (see the throughput path): the
// top bits of the bit pattern of max(f - lo + delta, 0), delta = (hi - lo) / 15,
// counted from those of delta; clamped to [0, kMBins).  Monotone in f.
struct LogBins {
  float d;          // delta - lo
  uint32_t base;    // bit pattern of delta
  __device__ __forceinline__ LogBins(float lo, float hi) {
    const float delta = (hi - lo) * (1.0f / 15.0f);
    d = delta - lo;
    base = __float_as_uint(delta);
  }
  __device__ __forceinline__ int operator()(float f) const {
    const int x = (int)(__float_as_uint(fmaxf(f + d, 0.0f)) - base) >> kLogShift;
    return min(max(x, 0), kMBins - 1);
  }
};

// Appends one batch's valid candidates (id >= 0) as raw (score, id) pairs and
// folds their score keys into [kmn, kmx] (no floor: the exact range).
__device__ __forceinline__ void append_valid(const float4 (&v)[kQuarter], MergeFastSmem& sm,
                                             int* counter, uint32_t& kmn, uint32_t& kmx) {
  const int lane = threadIdx.x & 31;
  uint32_t mask = 0u;
#pragma unroll
  for (int i = 0; i < kQuarter; ++i) {
    const bool a = __float_as_int(v[i].y) >= 0, b = __float_as_int(v[i].w) >= 0;
    mask |= (uint32_t)a << (2 * i);
    mask |= (uint32_t)b << (2 * i + 1);
    if (a) {
      kmn = min(kmn, score_key(v[i].x));
      kmx = max(kmx, score_key(v[i].x));
    }
    if (b) {
      kmn = min(kmn, score_key(v[i].z));
      kmx = max(kmx, score_key(v[i].z));
    }
  }
  const int m = __popc(mask);
  const int incl = warp_inclusive_scan(m);
  int base = 0;
  if (lane == 31 && incl) base = atomicAdd(counter, incl);
  int p = __shfl_sync(kFull, base, 31) + incl - m;
#pragma unroll
  for (int i = 0; i < kQuarter; ++i) {
    if ((mask >> (2 * i) & 1u) && p < kMListCap) sm.u.f[p] = make_float2(v[i].x, v[i].y);
    p += mask >> (2 * i) & 1u;
    if ((mask >> (2 * i + 1) & 1u) && p < kMListCap) sm.u.f[p] = make_float2(v[i].z, v[i].w);
    p += mask >> (2 * i + 1) & 1u;
  }
}

template <int NT>
__global__ void __launch_bounds__(NT, merge_fast_min_blocks<NT>())
    merge_fast_kernel(const float* __restrict__ cand, int C, int K, int32_t* __restrict__ ids,
                      float* __restrict__ scores) {
  extern __shared__ __align__(16) unsigned char merge_smem[];
  MergeFastSmem& sm = *reinterpret_cast<MergeFastSmem*>(merge_smem);
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = blockIdx.x;
  const float* row = cand + (int64_t)r * C * 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  int32_t* out_ids = ids + (int64_t)r * K;
  float* out_sc = scores ? scores + (int64_t)r * K : nullptr;

  // Float4 q = jj NT + tid holds elements 2 q and 2 q + 1 (C is a multiple of
  // 4, so a float4 holds two whole candidates or none).  Batch b holds rows
  // jj = 4 i + (i + b) mod 4.
  auto load_batch = [&](int b, float4 (&v)[kQuarter]) {
#pragma unroll
    for (int i = 0; i < kQuarter; ++i) {
      const int q = (4 * i + ((i + b) & 3)) * NT + tid;
      v[i] = 2 * q < C ? __ldg(row4 + q)
                       : make_float4(0.f, __int_as_float(-1), 0.f, __int_as_float(-1));
    }
  };
  float4 va[kQuarter], vb[kQuarter];
  load_batch(0, va);
  load_batch(1, vb);

  for (int b = tid; b < kSampBins; b += NT) sm.w.scnt[b] = 0u;
  for (int b = tid; b < kMBins; b += NT) sm.h.end[b] = 0u;
  if (tid == 0) {
    sm.nsv = 0;
    sm.nslots = 0;
    sm.nlist = 0;
    sm.nlist2 = 0;
    sm.nb = 0;
    sm.nwin = 0;   // the crowded path's winner count
    sm.bmax[0] = 0;
    sm.smin = 0xffffffffu;
    sm.smax = 0u;
    sm.lmin2 = 0xffffffffu;
    sm.kmax2 = 0u;
  }
  // Samples: one candidate of each float4 of batch 0, alternating halves.
  auto samp_f = [&](int i) { return (i & 1) ? va[i].z : va[i].x; };
  auto samp_ok = [&](int i) { return __float_as_int((i & 1) ? va[i].w : va[i].y) >= 0; };
  {
    int ns = 0, slots = 0;   // valid samples; sample positions inside the row
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int i = 0; i < kQuarter; ++i) {
      slots += 2 * (5 * i * NT + tid) < C;   // batch 0 holds rows 5 i
      if (samp_ok(i)) {
        const uint32_t k = score_key(samp_f(i));
        ++ns;
        mx = max(mx, k);
        mn = min(mn, k);
      }
    }
    ns = __reduce_add_sync(kFull, ns);
    slots = __reduce_add_sync(kFull, slots);
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    __syncthreads();
    if (lane == 0) {
      atomicAdd(&sm.nslots, slots);
      if (ns) {
        atomicAdd(&sm.nsv, ns);
        atomicMin(&sm.smin, mn);
        atomicMax(&sm.smax, mx);
      }
    }
  }
  __syncthreads();
  // The floor: the score above which about 1.125 K + 16 sample-equivalents lie.
  float ffloor = -INFINITY;   // -inf: no floor, every valid candidate is listed
  {
    const float smax_f = key_score(sm.smax);
    const int nsv = sm.nsv, nslots = sm.nslots;
    // Estimated valid candidates: the valid fraction of the sample slots times C.
    const float valid_est = nslots ? (float)nsv * (float)C / (float)nslots : 0.f;
    const float smin_f = key_score(sm.smin);
    constexpr float kTwo23 = 8388608.0f;
    const float scale = __fdividef((float)(kSampBins - 3), smax_f - smin_f);
    const LinearBinsN<kSampBins> sbin{scale, (kTwo23 + 1.0f) - smin_f * scale};
    // Same values in every thread: uniform.
    if (valid_est > 1.25f * (float)K && nsv >= 64 && smax_f > smin_f && isfinite(smin_f) &&
        isfinite(smax_f) && isfinite(scale) && sbin.v(smin_f) >= kTwo23 &&
        sbin.v(smax_f) <= kTwo23 + (float)(kSampBins - 1)) {
#pragma unroll
      for (int i = 0; i < kQuarter; ++i)
        if (samp_ok(i)) atomicAdd(&sm.w.scnt[sbin(samp_f(i))], 1u);
      __syncthreads();
      // Expected samples among the winners: K * nslots / C; take 1/8 more and 16.
      const int target = min(nsv, (int)((float)K * (float)nslots * 1.125f / (float)C) + 16);
      // Thread t < kSampBins takes bin kSampBins - 1 - t (bins from the top).
      const int local = tid < kSampBins ? (int)sm.w.scnt[kSampBins - 1 - tid] : 0;
      const int run = block_exclusive_scan_1bar(local, sm.scan);
      if (tid < kSampBins && run < target && run + local >= target) {
        // Bin b holds scores from about smin + (b - 1) / scale; one bin lower
        // for the rounding of the map.
        const int b = kSampBins - 1 - tid;
        sm.sfloor = b <= 2 ? smin_f : smin_f + (float)(b - 2) / scale;
      }
      __syncthreads();
      ffloor = sm.sfloor;
    }
  }

  int n = 0, need = 0;
  float lo = 0.f, hi = 0.f;
  if (ffloor > -INFINITY) {
    // Filter the four batches into the list, the next batch in flight meanwhile.
    append_batches(va, vb, ffloor, sm, &sm.nlist);
    load_batch(2, va);
    load_batch(3, vb);
    append_batches(va, vb, ffloor, sm, &sm.nlist);
    __syncthreads();
    n = sm.nlist;
    need = K;
    // Bins over [floor, largest sample]; the few above it share the top bin.
    lo = ffloor;
    hi = fmaxf(key_score(sm.smax), ffloor);
  }
  if (n < need || ffloor == -INFINITY) {
    // No floor, or it was above the K-th score: every valid candidate.
    uint32_t kmn = 0xffffffffu, kmx = 0u;
    for (int b = 0; b < 4; ++b) {
      load_batch(b, va);
      append_valid(va, sm, &sm.nlist2, kmn, kmx);
    }
    kmn = __reduce_min_sync(kFull, kmn);
    kmx = __reduce_max_sync(kFull, kmx);
    if (lane == 0 && kmn <= kmx) {
      atomicMin(&sm.lmin2, kmn);
      atomicMax(&sm.kmax2, kmx);
    }
    __syncthreads();
    n = sm.nlist2;
    need = min(K, n);
    lo = key_score(sm.lmin2);
    hi = key_score(sm.kmax2);
  }

  bool ranked = false;   // winners staged in out[] by position
  if (need > 0 && (n > kMListCap || !isfinite(lo) || !isfinite(hi))) {
    // Every winner's score is at or above lo; n valid candidates are.
    merge_crowded<NT>(row, C, score_key(lo), n, need, sm, out_ids, out_sc);
  } else if (need > 0) {
    const LogBins bin(lo, hi);
    for (int i = tid; i < n; i += NT) atomicAdd(&sm.h.end[bin(sm.u.f[i].x)], 1u);
    __syncthreads();
    // Scan from the top bin down: output ranges, b*, the largest bin above b*.
    {
      constexpr int per = kMBins / NT;
      const int g = kMBins - per * (tid + 1);
      int cnt[per];
      int local = 0;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        cnt[j] = (int)sm.h.end[g + per - 1 - j];
        local += cnt[j];
      }
      int run = block_exclusive_scan_1bar(local, sm.scan);
      int mx = 0;
#pragma unroll
      for (int j = 0; j < per; ++j) {
        const int b = g + per - 1 - j;
        sm.h.end[b] = (uint32_t)run;
        if (run < need && run + cnt[j] >= need) {
          sm.bstar = b;
          sm.above = run;
          sm.bcnt = cnt[j];
        } else if (run + cnt[j] < need) {
          mx = max(mx, cnt[j]);
        }
        run += cnt[j];
      }
      if (mx > kFineCap) atomicMax(&sm.bmax[0], mx);
    }
    __syncthreads();
    const int bstar = sm.bstar, above = sm.above, bcnt = sm.bcnt;
    ranked = bcnt <= kRankCap && sm.bmax[0] <= kFineCap;
    if (ranked) {
      const int take = need - above;   // members of b* that win
      // Winners above b* go to their bin's output range, b* to its own list.
      for (int i = tid; i < n; i += NT) {
        const float2 e = sm.u.f[i];
        const int b = bin(e.x);
        if (b < bstar) continue;
        const ull x = rank_key(e.x, e.y);
        if (b > bstar) sm.w.win[atomicAdd(&sm.h.end[b], 1u)] = x;
        else sm.bst[atomicAdd(&sm.nb, 1)] = x;
      }
      __syncthreads();
      for (int p = tid; p < above; p += NT) {
        const ull x = sm.w.win[p];
        // key_score(score_key(f)) is f (a -0.0 comes back as +0.0, which has
        // the same bin), so this is the bin the scatter used.
        const int b = bin(key_score((uint32_t)(x >> 32)));
        const int e = (int)sm.h.end[b], s0 = b == kMBins - 1 ? 0 : (int)sm.h.end[b + 1];
        sm.u.out[s0 + count_above<2>(sm.w.win, s0, e, x)] = x;
      }
      for (int i = tid; i < bcnt; i += NT) {
        const ull x = sm.bst[i];
        const int rank = count_above(sm.bst, 0, bcnt, x);
        if (rank < take) sm.u.out[above + rank] = x;
      }
      __syncthreads();
    } else {
      __syncthreads();   // the select reuses the bin counters
      merge_crowded<NT>(row, C, score_key(lo), n, need, sm, out_ids, out_sc);
    }
  }
  // Write the ranked winners and the -1 / -inf padding, 4 positions a thread.
  const bool vec = ((reinterpret_cast<uintptr_t>(out_ids) | reinterpret_cast<uintptr_t>(out_sc)) &
                    15u) == 0;
  const int first = ranked ? 0 : need;   // the crowded path wrote [0, need) itself
  for (int p0 = 4 * tid; p0 < K; p0 += 4 * NT) {
    if (p0 + 4 <= first) continue;
    int32_t oi[4];
    float os[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int p = p0 + u;
      if (ranked && p < need) {
        const ull x = sm.u.out[p];
        oi[u] = (int32_t)~(uint32_t)x;
        os[u] = key_score((uint32_t)(x >> 32));
      } else {
        oi[u] = -1;
        os[u] = -INFINITY;
      }
    }
    if (vec && p0 >= first) {
      *reinterpret_cast<int4*>(out_ids + p0) = make_int4(oi[0], oi[1], oi[2], oi[3]);
      if (out_sc) *reinterpret_cast<float4*>(out_sc + p0) = make_float4(os[0], os[1], os[2], os[3]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (p0 + u < first) continue;
        out_ids[p0 + u] = oi[u];
        if (out_sc) out_sc[p0 + u] = os[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Rows of up to 16 candidates per thread (C <= 16 NT; NT = 512 or 1024):
// every candidate stays in registers as (score key, ~id), so neither a floor
// nor a list is needed.  One pass gives the number of valid candidates and the
// range of their score keys; one 2048-bin histogram, the bins linear in the
// score over that range (monotone in the key: a rounded difference, a rounded
// positive product and a truncation never reverse two scores), and a scan from
// the top bin down give every bin above the bin b* of the need-th key its
// output range.  Winners above b* are scattered into those ranges and ranked
// inside their bins, b*'s members among themselves.  Rows with an infinite
// score, a single score value or crowded bins take merge_crowded.  Twice the
// threads of merge_fast_kernel per row: for batches that fit one wave, where a
// row's latency, not the throughput of many rows, sets the time.
// ---------------------------------------------------------------------------
constexpr int kLinPer = 16;   // candidates per thread

template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)
    merge_lin_kernel(const float* __restrict__ cand, int C, int K, int32_t* __restrict__ ids,
                     float* __restrict__ scores) {
  extern __shared__ __align__(16) unsigned char merge_smem[];
  MergeFastSmem& sm = *reinterpret_cast<MergeFastSmem*>(merge_smem);
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = blockIdx.x;
  const float* row = cand + (int64_t)r * C * 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  int32_t* out_ids = ids + (int64_t)r * K;
  float* out_sc = scores ? scores + (int64_t)r * K : nullptr;

  // Float4 q = j NT + tid holds candidates 2 q and 2 q + 1.
  uint32_t key[kLinPer], nid[kLinPer];   // score key (0: no candidate) and ~id
  {
    float4 v[kLinPer / 2];
#pragma unroll
    for (int j = 0; j < kLinPer / 2; ++j) {
      const int q = j * NT + tid;
      v[j] = 2 * q < C ? __ldg(row4 + q)
                       : make_float4(0.f, __int_as_float(-1), 0.f, __int_as_float(-1));
    }
#pragma unroll
    for (int j = 0; j < kLinPer / 2; ++j) {
      const int i0 = __float_as_int(v[j].y), i1 = __float_as_int(v[j].w);
      key[2 * j] = i0 >= 0 ? score_key(v[j].x) : 0u;
      key[2 * j + 1] = i1 >= 0 ? score_key(v[j].z) : 0u;
      nid[2 * j] = ~(uint32_t)i0;
      nid[2 * j + 1] = ~(uint32_t)i1;
    }
  }
  for (int b = tid; b < kMBins; b += NT) sm.h.end[b] = 0u;
  if (tid == 0) {
    sm.nlist = 0;
    sm.nb = 0;
    sm.nwin = 0;
    sm.bmax[0] = sm.bmax[1] = 0;
    sm.lmin = 0xffffffffu;
    sm.kmax = 0u;
  }
  {
    int nv = 0;
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (int i = 0; i < kLinPer; ++i)
      if (key[i]) {
        ++nv;
        mn = min(mn, key[i]);
        mx = max(mx, key[i]);
      }
    nv = __reduce_add_sync(kFull, nv);
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    __syncthreads();
    if (lane == 0 && nv) {
      atomicAdd(&sm.nlist, nv);
      atomicMin(&sm.lmin, mn);
      atomicMax(&sm.kmax, mx);
    }
  }
  __syncthreads();
  const int valid = sm.nlist;
  const int need = min(K, valid);
  bool ranked = false;   // winners ordered in out[] by position
  if (need > 0) {
    const float fmin = key_score(sm.lmin), fmax = key_score(sm.kmax);
    const float fscale = __fdividef((float)kMBins, fmax - fmin);
    // Same values in every thread: uniform.
    const bool lin = fmax > fmin && isfinite(fmin) && isfinite(fmax) && isfinite(fscale);
    auto bin = [&](uint32_t k) {
      return min(kMBins - 1, (int)__float2uint_rz((key_score(k) - fmin) * fscale));
    };
    if (lin) {
#pragma unroll
      for (int i = 0; i < kLinPer; ++i)
        if (key[i]) atomicAdd(&sm.h.end[bin(key[i])], 1u);
      __syncthreads();
      // Scan from the top bin down: output ranges, b*, the largest bin above b*.
      {
        constexpr int per = kMBins / NT;
        const int g = kMBins - per * (tid + 1);
        int cnt[per];
        int local = 0;
#pragma unroll
        for (int j = 0; j < per; ++j) {
          cnt[j] = (int)sm.h.end[g + per - 1 - j];
          local += cnt[j];
        }
        int run = block_exclusive_scan_1bar(local, sm.scan);
        int mx = 0;
#pragma unroll
        for (int j = 0; j < per; ++j) {
          const int b = g + per - 1 - j;
          sm.h.end[b] = (uint32_t)run;
          if (run < need && run + cnt[j] >= need) {
            sm.bstar = b;
            sm.above = run;
            sm.bcnt = cnt[j];
          } else if (run + cnt[j] < need) {
            mx = max(mx, cnt[j]);
          }
          run += cnt[j];
        }
        if (mx > kFineCap) atomicMax(&sm.bmax[0], mx);
      }
      __syncthreads();
      const int bstar = sm.bstar, above = sm.above, bcnt = sm.bcnt;
      ranked = bcnt <= kRankCap && sm.bmax[0] <= kFineCap;
      if (ranked) {
        const int take = need - above;   // members of b* that win
#pragma unroll
        for (int i = 0; i < kLinPer; ++i) {
          if (!key[i]) continue;
          const int b = bin(key[i]);
          const ull x = ((ull)key[i] << 32) | nid[i];
          if (b > bstar) sm.w.win[atomicAdd(&sm.h.end[b], 1u)] = x;
          else if (b == bstar) sm.bst[atomicAdd(&sm.nb, 1)] = x;
        }
        __syncthreads();
        for (int p = tid; p < above; p += NT) {
          const ull x = sm.w.win[p];
          const int b = bin((uint32_t)(x >> 32));
          const int e = (int)sm.h.end[b], s0 = b == kMBins - 1 ? 0 : (int)sm.h.end[b + 1];
          sm.u.out[s0 + count_above(sm.w.win, s0, e, x)] = x;
        }
        for (int i = tid; i < bcnt; i += NT) {
          const ull x = sm.bst[i];
          const int rank = count_above(sm.bst, 0, bcnt, x);
          if (rank < take) sm.u.out[above + rank] = x;
        }
        __syncthreads();
      }
    }
    if (!ranked) {
      __syncthreads();   // the select reuses the bin counters
      merge_crowded<NT>(row, C, 1u, valid, need, sm, out_ids, out_sc);
    }
  }
  // Write the ranked winners and the -1 / -inf padding, 4 positions a thread.
  const bool vec = ((reinterpret_cast<uintptr_t>(out_ids) | reinterpret_cast<uintptr_t>(out_sc)) &
                    15u) == 0;
  const int first = ranked ? 0 : need;   // the crowded path wrote [0, need) itself
  for (int p0 = 4 * tid; p0 < K; p0 += 4 * NT) {
    if (p0 + 4 <= first) continue;
    int32_t oi[4];
    float os[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int p = p0 + u;
      if (ranked && p < need) {
        const ull x = sm.u.out[p];
        oi[u] = (int32_t)~(uint32_t)x;
        os[u] = key_score((uint32_t)(x >> 32));
      } else {
        oi[u] = -1;
        os[u] = -INFINITY;
      }
    }
    if (vec && p0 >= first) {
      *reinterpret_cast<int4*>(out_ids + p0) = make_int4(oi[0], oi[1], oi[2], oi[3]);
      if (out_sc) *reinterpret_cast<float4*>(out_sc + p0) = make_float4(os[0], os[1], os[2], os[3]);
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (p0 + u < first) continue;
        out_ids[p0 + u] = oi[u];
        if (out_sc) out_sc[p0 + u] = os[u];
      }
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

dsa_status dsa::check_merge_topk_stable(const float* cand, int rows, int C, int K,
                                        const int32_t* ids) {
  if (rows < 0 || C < 0) return DSA_ERR_INVALID_ARG;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (C < K || (C & 3)) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!cand || !ids || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

extern "C" dsa_status dsa_merge_topk_stable(const float* cand, int rows, int C, int K,
                                            int32_t* ids, float* scores, uint32_t* err_flags,
                                            cudaStream_t stream) {
  const dsa_status st = check_merge_topk_stable(cand, rows, C, K, ids);
  if (st != DSA_OK || rows == 0) return st;
  if (C <= 32 * 1024) {
    auto launch_fast = [&](auto kernel, int nt) {
      const int smem = (int)sizeof(MergeFastSmem);
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return DSA_ERR_CUDA;
      const cudaError_t e = launch_kernel(kernel, dim3((unsigned)rows), dim3((unsigned)nt),
                                          (size_t)smem, stream, 0, cand, C, K, ids, scores);
      return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
    };
    // Batches that fit one wave are latency-bound: more threads per row
    // (1024 whenever a row per SM is enough, 512 for up to two rows per SM).
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (C <= kLinPer * 1024 && rows <= sms) return launch_fast(merge_lin_kernel<1024>, 1024);
    if (C <= kLinPer * 512 && rows <= 2 * sms) return launch_fast(merge_lin_kernel<512>, 512);
    if (C > kLinPer * 512 && C <= kLinPer * 1024 && rows <= sms)
      return launch_fast(merge_lin_kernel<1024>, 1024);
    if (C <= 32 * 256) return launch_fast(merge_fast_kernel<256>, 256);
    if (C <= 32 * 512) return launch_fast(merge_fast_kernel<512>, 512);
    return launch_fast(merge_fast_kernel<1024>, 1024);
  }
  (void)err_flags;   // no asynchronous copies on this path: nothing can stall
  const cudaError_t e = launch_kernel(merge_kernel, dim3((unsigned)rows), dim3(kMergeThreads), 0,
                                      stream, 0, cand, C, K, ids, scores);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
