// One shard's local top-K of one row, for one CTA (sm_103a).
//
// Staging of the local range into shared memory with bulk async copies, a
// radix select of the K-th best score key, and an ordered sweep that hands
// every winner, in ascending slot order, to a caller-supplied `emit`.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace dsa {

constexpr int kStageChunks = 16;
constexpr uint32_t kStageChunkBytes = 16384;
constexpr int kStageCapElems = 48 * 1024;  // 192 KB of staged logits at most

// DSA_TEST_STALLED_COPY (a separate test build, never libdsa.so): one more
// mbarrier, armed for 16 bytes that no copy delivers, joins the staging wait,
// so that the bounded wait runs out while every real copy still lands.
#ifdef DSA_TEST_STALLED_COPY
constexpr int kStageBars = kStageChunks + 1;
#else
constexpr int kStageBars = kStageChunks;
#endif

struct LocalTopkSmem {
  uint64_t bars[kStageBars];
  SelectSmem sel;
  int wgt[32], weq[32], eq_before[32], sel_before[32];
};

// Stage logits[lo, hi) of `row` (16-byte aligned, ld % 4 == 0, hi <= ld) into
// `stage`, rounding the range out to 16-byte boundaries (still inside the
// row).  Returns the pointer the select should read: the staged copy, or the
// global row itself when the range is longer than `stage_cap`.  On a stalled
// copy it raises DSA_FLAG_TIMEOUT, waits once more (bounded) and sets *ok = false.
// Every thread must call it.
__device__ __forceinline__ const float* stage_local_range(const float* row, int64_t lo,
                                                          int64_t hi, float* stage,
                                                          int stage_cap, LocalTopkSmem& sm,
                                                          uint32_t* flags, bool* ok) {
  *ok = true;
  const int64_t lo4 = lo & ~int64_t(3), hi4 = (hi + 3) & ~int64_t(3);
  if (hi4 - lo4 > stage_cap) return row + lo;
  const uint32_t bytes = (uint32_t)((hi4 - lo4) * 4);
  const int nchunks = (int)((bytes + kStageChunkBytes - 1) / kStageChunkBytes);
  if (threadIdx.x == 0) {
    for (int c = 0; c < nchunks; ++c) mbar_init(&sm.bars[c], 1);
#ifdef DSA_TEST_STALLED_COPY
    mbar_init(&sm.bars[kStageChunks], 1);
#endif
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t off = c * kStageChunkBytes;
      const uint32_t len = min(kStageChunkBytes, bytes - off);
      mbar_expect_tx(&sm.bars[c], len);
      bulk_g2s(reinterpret_cast<unsigned char*>(stage) + off,
               reinterpret_cast<const unsigned char*>(row + lo4) + off, len, &sm.bars[c]);
    }
  }
#ifdef DSA_TEST_STALLED_COPY
  if (threadIdx.x == 0) mbar_expect_tx(&sm.bars[kStageChunks], 16);
#endif
  bool good = true;
  for (int c = 0; c < nchunks; ++c) good &= mbar_wait(&sm.bars[c], 0);
#ifdef DSA_TEST_STALLED_COPY
  good &= mbar_wait(&sm.bars[kStageChunks], 0);
#endif
  if (__syncthreads_or(!good)) {
    if (threadIdx.x == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
    for (int c = 0; c < nchunks; ++c) mbar_wait(&sm.bars[c], 0);
    *ok = false;
  }
  return stage + (lo - lo4);
}

// The K best of data[0, n) (n > K) under (score desc, index asc), handed to
// emit(p, i, v) with p = 0..K-1 in ascending i.  NT threads; ends with all
// emits issued (no trailing barrier).
template <int NT, typename Emit>
__device__ __forceinline__ void local_topk_emit(const float* data, int n, int K,
                                                LocalTopkSmem& sm, Emit emit) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  auto key_at = [&](int i, uint32_t& k) {
    k = score_key(data[i]);
    return true;
  };
  const SelectResult res = radix_select<NT>(n, K, key_at, sm.sel);
  const uint32_t thr = res.thr;
  const int take_eq = res.take_eq;

  // Warp w owns the contiguous indices [w*seg, w*seg + seg).
  const int seg = (((n + kWarps - 1) / kWarps) + 31) & ~31;
  const int w_lo = min(n, warp * seg), w_hi = min(n, w_lo + seg);
  int gt = 0, eq = 0;
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    const bool in = i < w_hi;
    const uint32_t k = in ? score_key(data[i]) : 0u;
    gt += __popc(__ballot_sync(kFull, in && k > thr));
    eq += __popc(__ballot_sync(kFull, in && k == thr));
  }
  if (lane == 0) { sm.wgt[warp] = gt; sm.weq[warp] = eq; }
  __syncthreads();
  if (warp == 0) {
    const int g = lane < kWarps ? sm.wgt[lane] : 0;
    const int e = lane < kWarps ? sm.weq[lane] : 0;
    int e_incl = e;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, e_incl, o);
      if (lane >= o) e_incl += y;
    }
    const int e_before = e_incl - e;
    const int take = g + max(0, min(take_eq - e_before, e));
    int t_incl = take;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, t_incl, o);
      if (lane >= o) t_incl += y;
    }
    if (lane < kWarps) { sm.eq_before[lane] = e_before; sm.sel_before[lane] = t_incl - take; }
  }
  __syncthreads();
  int eq_seen = sm.eq_before[warp], pos = sm.sel_before[warp];
  const unsigned lt = lanemask_lt();
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    const bool in = i < w_hi;
    const float v = in ? data[i] : 0.f;
    const uint32_t k = in ? score_key(v) : 0u;
    const bool is_gt = in && k > thr, is_eq = in && k == thr;
    const unsigned eqm = __ballot_sync(kFull, is_eq);
    const bool sel = is_gt || (is_eq && eq_seen + __popc(eqm & lt) < take_eq);
    const unsigned selm = __ballot_sync(kFull, sel);
    const int p = pos + __popc(selm & lt);
    if (sel && p < K) emit(p, i, v);
    pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
}

}  // namespace dsa
