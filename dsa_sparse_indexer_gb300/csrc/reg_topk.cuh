// Register-resident local top-K of one row range for one CTA (sm_103a).
//
// Each of the NT threads loads VEC float4 vectors of the range with 16-byte
// loads and keeps their order-preserving score keys in registers: element e
// (counted from the 16-byte aligned start `base` = lo & ~3) lives in thread
// (e / 4) mod NT, vector (e / 4) / NT, lane c = e mod 4.  Positions outside
// [lo, hi) hold key 0, which no score maps to.  The radix select then reads
// registers only, and the winners are emitted in ascending e by warp ballots
// over (vector, warp) groups with one block-wide scan.
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace dsa {

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

// Emit the winners of a select over register keys in ascending element order:
// emit(p, e, k) with p = 0, 1, ... (output position), e = element index from
// base, k = its key.  An element wins if k > thr, or k == thr and fewer than
// take_eq elements with key thr come before it.
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
      e += key[j][c] == thr;
    }
    cg[j] = g;
    ce[j] = e;
    const int ie = warp_inclusive_scan(e);
    const int ig = warp_inclusive_scan(g);
    pe[j] = ie - e;
    if (lane == 31) {
      es.eq[j * R::kWarps + warp] = ie;
      es.gt[j * R::kWarps + warp] = ig;
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
    int pos = es.sel_before[grp] + warp_inclusive_scan(nsel) - nsel;
    const int e0 = (j * NT + (int)threadIdx.x) * 4;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t k = key[j][c];
      bool sel = k > thr;
      if (k == thr) {
        sel = eqb < take_eq;
        ++eqb;
      }
      if (sel) emit(pos++, e0 + c, k);
    }
  }
}

}  // namespace dsa
