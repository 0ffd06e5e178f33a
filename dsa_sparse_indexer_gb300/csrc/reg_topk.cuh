// Register-resident local top-K of one row range for one CTA (sm_103a).
//
// Each of the NT threads loads VEC float4 vectors of the range with 16-byte
// loads and keeps their order-preserving score keys in registers: element e
// (counted from the 16-byte aligned start `base` = lo & ~3) lives in thread
// (e / 4) mod NT, vector (e / 4) / NT, lane c = e mod 4.  Positions outside
// [lo, hi) hold key 0, which no score maps to.
//
// Selection: the first digit is histogrammed from registers; the keys of the
// bin holding the K-th key (typically a few percent of the range) are then
// compacted into a shared list, and the remaining digits run on that list.
// Emission hands the winners to a callback either in ascending element order
// (warp ballots over (vector, warp) groups and one block-wide scan), or, when
// the order does not matter and no tie has to be broken by position, with one
// counting pass and a warp-aggregated append.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace dsa {

constexpr int kListCap = 4096;   // keys of the threshold bin compacted to shared memory

template <int NT, int VEC>
struct RegTopk {
  static constexpr int kWarps = NT / 32;
  static constexpr int kGroups = VEC * kWarps;   // (vector, warp) groups, in element order
  static constexpr int64_t kCap = (int64_t)NT * VEC * 4;
  static_assert(kGroups % 32 == 0, "one warp scans the group counts");
};

template <int NT, int VEC>
struct RegEmitSmem {
  int gt[RegTopk<NT, VEC>::kGroups];
  int eq[RegTopk<NT, VEC>::kGroups];
  int eq_before[RegTopk<NT, VEC>::kGroups];
  int sel_before[RegTopk<NT, VEC>::kGroups];
  int nlist;     // entries in the compacted list
  int nout;      // winners appended by the unordered emission
};

// Keys of row[lo, hi) into registers.  Requires hi - (lo & ~3) <= kCap, a
// 16-byte aligned row and hi <= the row's allocated length rounded up to 4.
template <int NT, int VEC>
__device__ __forceinline__ void load_keys(const float* __restrict__ row, int64_t lo, int64_t hi,
                                          uint32_t (&key)[VEC][4]) {
  const int64_t base = lo & ~int64_t(3);
  float4 v[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int64_t e0 = base + ((int64_t)j * NT + threadIdx.x) * 4;
    v[j] = e0 < hi ? __ldg(reinterpret_cast<const float4*>(row + e0))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int64_t e0 = base + ((int64_t)j * NT + threadIdx.x) * 4;
    const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int c = 0; c < 4; ++c) key[j][c] = (e0 + c >= lo && e0 + c < hi) ? score_key(f[c]) : 0u;
  }
}

__device__ __forceinline__ int warp_inclusive_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive warp prefix of a small count 0 <= v < 8 from three ballots.
__device__ __forceinline__ int warp_scan_small(int v, int* total) {
  const unsigned lt = lanemask_lt();
  const unsigned b0 = __ballot_sync(kFull, v & 1), b1 = __ballot_sync(kFull, v & 2),
                 b2 = __ballot_sync(kFull, v & 4);
  *total = __popc(b0) + 2 * __popc(b1) + 4 * __popc(b2);
  return __popc(b0 & lt) + 2 * __popc(b1 & lt) + 4 * __popc(b2 & lt);
}

// The need-th largest key among the register keys (1 <= need < number of keys).
// `list` holds LIST_CAP keys of shared memory; *nlist is a shared counter.
// *eq as radix_select_from.
template <int NT, int VEC, int LIST_CAP = kListCap>
__device__ SelectResult select_regs_into(const uint32_t (&key)[VEC][4], int need, SelectSmem& sm,
                                         uint32_t* list, int* nlist, int* eq) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int b = tid; b < 2048; b += NT) sm.hist[b] = 0u;
  if (tid == 0) *nlist = 0;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (key[j][c]) atomicAdd(&sm.hist[key[j][c] >> 21], 1u);
  __syncthreads();
  find_bin<NT, 2048>(need, sm);
  const uint32_t b = (uint32_t)sm.bin;
  const int count = sm.count;
  need -= sm.above;
  *eq = count;
  if (count == need) return SelectResult{(b << 21) - 1u, 0};
  const uint32_t prefix = b << 21, mask = 0x7ffu << 21;
  if (count <= LIST_CAP) {
    int mine = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) mine += key[j][c] && (key[j][c] & mask) == prefix;
    const int incl = warp_inclusive_scan(mine);
    int base = 0;
    if (lane == 31 && incl) base = atomicAdd(nlist, incl);
    int p = __shfl_sync(kFull, base, 31) + incl - mine;
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (key[j][c] && (key[j][c] & mask) == prefix) list[p++] = key[j][c];
    __syncthreads();
    auto visit = [&](auto&& f) {
      for (int i = tid; i < count; i += NT) f(list[i]);
    };
    return radix_select_from<NT>(1, prefix, mask, need, visit, sm, eq);
  }
  auto visit = [&](auto&& f) {
#pragma unroll
    for (int j = 0; j < VEC; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (key[j][c]) f(key[j][c]);
  };
  return radix_select_from<NT>(1, prefix, mask, need, visit, sm, eq);
}

template <int NT, int VEC>
__device__ __forceinline__ SelectResult select_regs(const uint32_t (&key)[VEC][4], int need,
                                                    SelectSmem& sm, uint32_t* list,
                                                    RegEmitSmem<NT, VEC>& es, int* eq) {
  return select_regs_into<NT, VEC>(key, need, sm, list, &es.nlist, eq);
}

// Winners in any order: every key >= lo_key (the caller has made sure no tie
// needs breaking).  emit(p, e, k) with distinct p = 0, 1, ...; es.nout must be
// zero and visible to all threads.
template <int NT, int VEC, typename Emit>
__device__ __forceinline__ void emit_unordered(const uint32_t (&key)[VEC][4], uint32_t lo_key,
                                               RegEmitSmem<NT, VEC>& es, Emit emit) {
  const int lane = threadIdx.x & 31;
  int mine = 0;
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) mine += key[j][c] >= lo_key;
  const int incl = warp_inclusive_scan(mine);
  int base = 0;
  if (lane == 31 && incl) base = atomicAdd(&es.nout, incl);
  int p = __shfl_sync(kFull, base, 31) + incl - mine;
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (key[j][c] >= lo_key) emit(p++, (j * NT + (int)threadIdx.x) * 4 + c, key[j][c]);
}

// Winners in ascending element order: emit(p, e, k) with p = 0, 1, ...  An
// element wins if k > thr, or k == thr and fewer than take_eq elements with key
// thr come before it.
template <int NT, int VEC, typename Emit>
__device__ __forceinline__ void emit_winners(const uint32_t (&key)[VEC][4], uint32_t thr,
                                             int take_eq, RegEmitSmem<NT, VEC>& es, Emit emit) {
  using R = RegTopk<NT, VEC>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cg[VEC], ce[VEC], pe[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    int g = 0, e = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      g += key[j][c] > thr;
      e += key[j][c] && key[j][c] == thr;
    }
    cg[j] = g;
    ce[j] = e;
    int te, tg;
    pe[j] = warp_scan_small(e, &te);
    warp_scan_small(g, &tg);
    if (lane == 0) {
      es.eq[j * R::kWarps + warp] = te;
      es.gt[j * R::kWarps + warp] = tg;
    }
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int per = R::kGroups / 32;   // consecutive groups per lane
    int e_loc = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) e_loc += es.eq[lane * per + q];
    int e_run = warp_inclusive_scan(e_loc) - e_loc;
    int take_loc[per];
    int t_sum = 0;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      const int idx = lane * per + q;
      const int e = es.eq[idx];
      es.eq_before[idx] = e_run;
      take_loc[q] = es.gt[idx] + max(0, min(take_eq - e_run, e));
      t_sum += take_loc[q];
      e_run += e;
    }
    int t_run = warp_inclusive_scan(t_sum) - t_sum;
#pragma unroll
    for (int q = 0; q < per; ++q) {
      es.sel_before[lane * per + q] = t_run;
      t_run += take_loc[q];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int grp = j * R::kWarps + warp;
    int eqb = es.eq_before[grp] + pe[j];
    const int nsel = cg[j] + max(0, min(take_eq - eqb, ce[j]));
    int tsel;
    int pos = es.sel_before[grp] + warp_scan_small(nsel, &tsel);
    const int e0 = (j * NT + (int)threadIdx.x) * 4;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t k = key[j][c];
      bool sel = k > thr;
      if (k && k == thr) {
        sel = eqb < take_eq;
        ++eqb;
      }
      if (sel) emit(pos++, e0 + c, k);
    }
  }
}

}  // namespace dsa
