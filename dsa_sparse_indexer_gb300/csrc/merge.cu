// Stable global top-K of the gathered (score, global id) candidates.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 实现拆解 item 1 (`stable_topk_from_gathered_candidates_cutedsl`, a
// radix selector) and section 关键源码片段 (the all_gathered [batch, S*topk, 2]
// buffer; topk_indices overwritten with global ids, -1 for padding).
//
// One CTA per row.  The row's C candidates are staged in shared memory by bulk
// async copies.  Selection is a radix select on the score key, and, only when
// the K-th score is tied, a second radix select on the inverted id among the
// tied candidates (ties go to the smaller id).  The K winners are then put in
// rank order by a bitonic sort of their 64-bit keys (score_key << 32 | ~id).
#include "common.cuh"
#include "reg_topk.cuh"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kMergeThreads = 1024;
constexpr int kMaxChunks = 16;
constexpr uint32_t kChunkBytes = 16384;
constexpr int kStageCapCand = 20 * 1024;   // 160 KB of staged candidates at most
constexpr int kMaxK = 2048;

struct MergeSmem {
  uint64_t bars[kMaxChunks];
  SelectSmem sel;
  unsigned long long win[kMaxK];
  int nwin;
  int valid_count;
  int tied;
};

__host__ __device__ constexpr size_t merge_stage_offset() {
  return (sizeof(MergeSmem) + 127) & ~size_t(127);
}

__global__ void __launch_bounds__(kMergeThreads, 1)
    merge_kernel(const float* __restrict__ cand, int C, int K, int32_t* __restrict__ ids,
                 float* __restrict__ scores, uint32_t* flags, int stage_cap) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MergeSmem& sm = *reinterpret_cast<MergeSmem*>(smem_raw);
  float2* stage = reinterpret_cast<float2*>(smem_raw + merge_stage_offset());
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = blockIdx.x;
  const float2* row = reinterpret_cast<const float2*>(cand) + (int64_t)r * C;
  const float2* data = row;

  if (tid == 0) { sm.nwin = 0; sm.valid_count = 0; sm.tied = 0; }
  __syncthreads();
  if (C <= stage_cap) {
    const uint32_t bytes = (uint32_t)C * 8u;
    const int nchunks = (int)((bytes + kChunkBytes - 1) / kChunkBytes);
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) mbar_init(&sm.bars[c], 1);
      mbar_init_fence();
    }
    __syncthreads();
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) {
        const uint32_t off = c * kChunkBytes;
        const uint32_t len = min(kChunkBytes, bytes - off);
        mbar_expect_tx(&sm.bars[c], len);
        bulk_g2s(reinterpret_cast<unsigned char*>(stage) + off,
                 reinterpret_cast<const unsigned char*>(row) + off, len, &sm.bars[c]);
      }
    }
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) ok &= mbar_wait(&sm.bars[c], 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
      for (int c = 0; c < nchunks; ++c) mbar_wait(&sm.bars[c], 0);
      return;
    }
    data = stage;
  }

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
// Throughput path (C <= 32 * NT): each thread keeps 32 candidates' score keys
// in registers; a radix select with threshold-bin compaction (reg_topk.cuh)
// finds the K-th score, ties on it are broken by a select on ~id (ids
// reloaded from L2); the winners' 64-bit rank keys are then put in order by a
// 1024-bin counting sort over their score range plus a sort inside each (small)
// bin, and written straight to their output positions.  Rows whose winners
// crowd a bin (heavy ties) are sorted by a bitonic network instead.  Small
// shared memory and 64 registers per thread keep 1024 / NT rows per SM.
// ---------------------------------------------------------------------------
using ull = unsigned long long;
constexpr int kFineBins = 1024;
constexpr int kFineCap = 64;          // larger bins take the bitonic sort
constexpr int kFastListCap = 2048;
constexpr int kFastVec = 8;           // 32 candidates per thread

struct MergeFastSmem {
  SelectSmem sel;
  uint32_t off[kFineBins], end[kFineBins];
  ull win[kMaxK];
  union {
    uint32_t list[kFastListCap];      // threshold-bin keys during the select
    ull lb[kMaxK];                    // winners in bin order
  } u;
  int nlist, nwin, nvalid, bmax;
  uint32_t kmin, kmax;
};

template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)
    merge_fast_kernel(const float* __restrict__ cand, int C, int K, int32_t* __restrict__ ids,
                      float* __restrict__ scores) {
  __shared__ __align__(16) MergeFastSmem sm;
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = blockIdx.x;
  const float4* row4 = reinterpret_cast<const float4*>(cand + (int64_t)r * C * 2);
  const int32_t* rowi = reinterpret_cast<const int32_t*>(cand + (int64_t)r * C * 2);
  if (tid == 0) {
    sm.nwin = 0;
    sm.nvalid = 0;
    sm.bmax = 0;
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
  }

  // Candidate u of this thread: float4 q = (u / 2) * NT + tid, half u % 2;
  // element e = 2 q + u % 2.
  // C is a multiple of 4, so a float4 holds two whole candidates or none.
  uint32_t key[kFastVec][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    constexpr int kHalf = kFastVec;
    float4 v[kHalf];
#pragma unroll
    for (int j = 0; j < kHalf; ++j) {
      const int q = (h * kHalf + j) * NT + tid;
      v[j] = 2 * q < C ? __ldg(row4 + q)
                       : make_float4(0.f, __int_as_float(-1), 0.f, __int_as_float(-1));
    }
#pragma unroll
    for (int j = 0; j < kHalf; ++j) {
      const int jj = h * kHalf + j;
      key[jj >> 1][(jj & 1) * 2] = __float_as_int(v[j].y) >= 0 ? score_key(v[j].x) : 0u;
      key[jj >> 1][(jj & 1) * 2 + 1] = __float_as_int(v[j].w) >= 0 ? score_key(v[j].z) : 0u;
    }
  }
  int nv = 0;
#pragma unroll
  for (int j = 0; j < kFastVec; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) nv += key[j][c] != 0u;
  nv = __reduce_add_sync(kFull, nv);
  __syncthreads();
  if (lane == 0 && nv) atomicAdd(&sm.nvalid, nv);
  __syncthreads();
  const int valid = sm.nvalid;
  auto elem = [&](int j, int c) { return 2 * ((2 * j + (c >> 1)) * NT + tid) + (c & 1); };

  // Winner rule: key > thr, or key == thr and (!tie or ~id >= thr2).
  uint32_t thr = 0u, thr2 = 0u;
  bool eq_in = false, tie = false;
  if (valid > K) {
    int eq;
    const SelectResult res = select_regs_into<NT, kFastVec, kFastListCap>(key, K, sm.sel, sm.u.list,
                                                                          &sm.nlist, &eq);
    thr = res.thr;
    if (res.take_eq > 0) {
      eq_in = true;
      if (res.take_eq < eq) {
        auto visit = [&](auto&& f) {
#pragma unroll
          for (int j = 0; j < kFastVec; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (key[j][c] == thr) f(~(uint32_t)__ldg(rowi + 2 * elem(j, c) + 1));
        };
        const SelectResult b = radix_select_visit<NT>(res.take_eq, visit, sm.sel);
        thr2 = b.take_eq > 0 ? b.thr : b.thr + 1u;
        tie = true;
      }
    }
  } else {
    eq_in = true;   // thr = 0 and key 0 marks padding: every valid candidate wins
    thr = 1u;
  }
  __syncthreads();

  // Gather the winners' 64-bit rank keys (any order) and their score range.
  {
    uint32_t wins = 0u;   // bit 4 j + c: key[j][c] wins
#pragma unroll
    for (int j = 0; j < kFastVec; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t k = key[j][c];
        bool w = k > thr || (eq_in && k == thr && k != 0u);
        if (tie && k == thr && ~(uint32_t)__ldg(rowi + 2 * elem(j, c) + 1) < thr2) w = false;
        wins |= (uint32_t)w << (4 * j + c);
      }
    const int mine = __popc(wins);
    uint32_t kmn = 0xffffffffu, kmx = 0u;
    const int incl = warp_inclusive_scan(mine);
    int base = 0;
    if (lane == 31 && incl) base = atomicAdd(&sm.nwin, incl);
    int p = __shfl_sync(kFull, base, 31) + incl - mine;
#pragma unroll
    for (int j = 0; j < kFastVec; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t k = key[j][c];
        if (wins >> (4 * j + c) & 1u) {
          const uint32_t nid = ~(uint32_t)__ldg(rowi + 2 * elem(j, c) + 1);
          if (p < kMaxK) sm.win[p] = ((ull)k << 32) | nid;
          ++p;
          kmn = min(kmn, k);
          kmx = max(kmx, k);
        }
      }
    kmn = __reduce_min_sync(kFull, kmn);
    kmx = __reduce_max_sync(kFull, kmx);
    if (lane == 0) {
      atomicMin(&sm.kmin, kmn);
      atomicMax(&sm.kmax, kmx);
    }
  }
  __syncthreads();
  const int nwin = min(sm.nwin, K);
  int32_t* out_ids = ids + (int64_t)r * K;
  float* out_sc = scores ? scores + (int64_t)r * K : nullptr;

  // 1024-bin counting sort of the winners by score key, highest bin first.
  const uint32_t kmin = sm.kmin;
  int sh = 0;
  while (((sm.kmax - kmin) >> sh) >= (uint32_t)kFineBins) ++sh;
  for (int b = tid; b < kFineBins; b += NT) sm.end[b] = 0u;
  __syncthreads();
  for (int i = tid; i < nwin; i += NT)
    atomicAdd(&sm.end[((uint32_t)(sm.win[i] >> 32) - kmin) >> sh], 1u);
  __syncthreads();
  {
    constexpr int per = kFineBins / NT;
    const int g = kFineBins - per * (tid + 1);
    int c[per];
    int local = 0, mx = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) {
      c[j] = (int)sm.end[g + per - 1 - j];
      local += c[j];
      mx = max(mx, c[j]);
    }
    int tot;
    int run = block_exclusive_scan(local, sm.sel.scan, &tot);
#pragma unroll
    for (int j = 0; j < per; ++j) {
      const int b = g + per - 1 - j;
      sm.off[b] = (uint32_t)run;
      sm.end[b] = (uint32_t)run;
      run += c[j];
    }
    if (mx > kFineCap) atomicMax(&sm.bmax, mx);
  }
  __syncthreads();
  if (sm.bmax <= kFineCap) {
    for (int i = tid; i < nwin; i += NT) {
      const ull x = sm.win[i];
      sm.u.lb[atomicAdd(&sm.end[((uint32_t)(x >> 32) - kmin) >> sh], 1u)] = x;
    }
    __syncthreads();
    for (int p = tid; p < nwin; p += NT) {
      const ull x = sm.u.lb[p];
      const int b = (int)(((uint32_t)(x >> 32) - kmin) >> sh);
      int pos = (int)sm.off[b];
      for (uint32_t q = sm.off[b]; q < sm.end[b]; ++q) pos += sm.u.lb[q] > x;
      out_ids[pos] = (int32_t)~(uint32_t)x;
      if (out_sc) out_sc[pos] = key_score((uint32_t)(x >> 32));
    }
  } else {
    // Heavy ties: a descending bitonic sort of the winners padded with 0 to
    // a power of two (at most kMaxK).
    int P = 1;
    while (P < nwin) P <<= 1;
    for (int j = nwin + tid; j < P; j += NT) sm.win[j] = 0ull;
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int p = tid; p < (P >> 1); p += NT) {
          const int i = 2 * p - (p & (j - 1));
          const int ixj = i + j;
          const bool desc = (i & k) == 0;
          const ull a = sm.win[i], b = sm.win[ixj];
          if ((a < b) == desc) { sm.win[i] = b; sm.win[ixj] = a; }
        }
        __syncthreads();
      }
    }
    for (int p = tid; p < nwin; p += NT) {
      const ull x = sm.win[p];
      out_ids[p] = (int32_t)~(uint32_t)x;
      if (out_sc) out_sc[p] = key_score((uint32_t)(x >> 32));
    }
  }
  for (int j = nwin + tid; j < K; j += NT) {
    out_ids[j] = -1;
    if (out_sc) out_sc[j] = -INFINITY;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_merge_topk_stable(const float* cand, int rows, int C, int K,
                                            int32_t* ids, float* scores, uint32_t* err_flags,
                                            cudaStream_t stream) {
  if (rows < 0 || C < 0) return DSA_ERR_INVALID_ARG;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (C < K || (C & 3)) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!cand || !ids || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  if (C <= 32 * 256) {
    const cudaError_t e = launch_kernel(merge_fast_kernel<256>, dim3((unsigned)rows), dim3(256), 0,
                                        stream, 0, cand, C, K, ids, scores);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (C <= 32 * 512) {
    const cudaError_t e = launch_kernel(merge_fast_kernel<512>, dim3((unsigned)rows), dim3(512), 0,
                                        stream, 0, cand, C, K, ids, scores);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (C <= 32 * 1024) {
    const cudaError_t e = launch_kernel(merge_fast_kernel<1024>, dim3((unsigned)rows), dim3(1024),
                                        0, stream, 0, cand, C, K, ids, scores);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  const int stage_cap = kStageCapCand;
  const size_t smem = merge_stage_offset() + (size_t)min(C, stage_cap) * sizeof(float2);
  if (cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const cudaError_t e = launch_kernel(merge_kernel, dim3((unsigned)rows), dim3(kMergeThreads), smem,
                                      stream, 0, cand, C, K, ids, scores, err_flags, stage_cap);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
