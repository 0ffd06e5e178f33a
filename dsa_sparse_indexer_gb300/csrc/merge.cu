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
  const int stage_cap = kStageCapCand;
  const size_t smem = merge_stage_offset() + (size_t)min(C, stage_cap) * sizeof(float2);
  if (cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  merge_kernel<<<rows, kMergeThreads, smem, stream>>>(cand, C, K, ids, scores, err_flags,
                                                      stage_cap);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
