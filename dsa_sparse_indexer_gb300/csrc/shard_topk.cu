// Per-shard local top-K of fp32 indexer logits, and candidate packing.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE":
// section 关键源码片段 (`_merge_dcp_topk_global`: the local top-K positions of
// each rank, then (score, global_id) candidates packed as [batch, topk, 2]
// fp32) and section 实现拆解 item 1 (`pack_dcp_topk_candidates_cutedsl`).
//
// One CTA per (shard, row).  The row's local range is staged in shared memory
// with bulk async copies (TMA), a radix select finds the K-th best score key,
// and one ordered sweep with warp ballots writes the winners in ascending slot
// order (ties on the score go to the smaller slot, i.e. the smaller global id).
#include "common.cuh"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kMaxChunks = 16;
constexpr uint32_t kChunkBytes = 16384;
constexpr int kStageCapElems = 48 * 1024;  // 192 KB of staged logits at most

struct TopkSmem {
  uint64_t bars[kMaxChunks];
  SelectSmem sel;
  int wgt[32], weq[32], eq_before[32], sel_before[32];
};

__host__ __device__ constexpr size_t topk_stage_offset() {
  return (sizeof(TopkSmem) + 127) & ~size_t(127);
}

__device__ __forceinline__ void write_pad(int32_t* out_idx, float2* out_cand, int j) {
  if (out_idx) out_idx[j] = -1;
  if (out_cand) out_cand[j] = make_float2(-INFINITY, __int_as_float(-1));
}

template <bool kPack>
__global__ void __launch_bounds__(kTopkThreads, 2)
    shard_topk_kernel(const float* __restrict__ logits, int64_t ld, int rows, int S, int I,
                      int K, const int32_t* __restrict__ row_starts,
                      const int32_t* __restrict__ row_ends, int32_t* __restrict__ local_idx,
                      float* __restrict__ cand, uint32_t* flags, int stage_cap) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  float* stage = reinterpret_cast<float*>(smem_raw + topk_stage_offset());

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x / rows, r = blockIdx.x - s * rows;
  const float* row = logits + ((int64_t)s * rows + r) * ld;

  // Global range -> this shard's local range.
  int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  int64_t lo = local_len(st, s, S, I), hi = local_len(en, s, S, I);
  if (hi > ld) { hi = ld; bad = true; }
  if (lo > hi) { lo = hi; bad = true; }
  if (bad && tid == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
  const int n = (int)(hi - lo);

  int32_t* out_idx = local_idx ? local_idx + ((int64_t)s * rows + r) * K : nullptr;
  float2* out_cand = kPack ? reinterpret_cast<float2*>(cand) + ((int64_t)r * S + s) * K : nullptr;

  if (n <= K) {  // every slot is selected: slots lo..hi-1 in order, then padding
    for (int j = tid; j < K; j += kTopkThreads) {
      if (j < n) {
        const int64_t l = lo + j;
        if (out_idx) out_idx[j] = (int32_t)l;
        if (kPack) out_cand[j] = make_float2(row[l], __int_as_float((int)global_of(s, l, S, I)));
      } else {
        write_pad(out_idx, out_cand, j);
      }
    }
    return;
  }

  // Stage [lo4, hi4) (16-byte aligned: the row base is aligned and ld % 4 == 0).
  const int64_t lo4 = lo & ~int64_t(3), hi4 = (hi + 3) & ~int64_t(3);
  const bool staged = (hi4 - lo4) <= stage_cap;
  const float* data = row + lo;
  if (staged) {
    const uint32_t bytes = (uint32_t)((hi4 - lo4) * 4);
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
                 reinterpret_cast<const unsigned char*>(row + lo4) + off, len, &sm.bars[c]);
      }
    }
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) ok &= mbar_wait(&sm.bars[c], 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
      for (int c = 0; c < nchunks; ++c) mbar_wait(&sm.bars[c], 0);
      return;
    }
    data = stage + (lo - lo4);
  }

  auto key_at = [&](int i, uint32_t& k) {
    k = score_key(data[i]);
    return true;
  };
  const SelectResult res = radix_select<kTopkThreads>(n, K, key_at, sm.sel);
  const uint32_t thr = res.thr;
  const int take_eq = res.take_eq;

  // Ordered emission.  Warp w owns the contiguous slots [w*seg, w*seg + seg).
  constexpr int kWarps = kTopkThreads / 32;
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
    if (sel && pos + __popc(selm & lt) < K) {
      const int p = pos + __popc(selm & lt);
      const int64_t l = lo + i;
      if (out_idx) out_idx[p] = (int32_t)l;
      if (kPack) out_cand[p] = make_float2(v, __int_as_float((int)global_of(s, l, S, I)));
    }
    pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
}

// Standalone pack: cand[r][s*K + j] from local_idx[s][r][j].  Each thread
// handles four consecutive j (K % 4 == 0): one 16-byte index load, four
// gathers from the logits, two 16-byte candidate stores.
__global__ void __launch_bounds__(256)
    pack_kernel(const float* __restrict__ logits, int64_t ld,
                const int32_t* __restrict__ local_idx, int rows, int S, int I, int K,
                float* __restrict__ cand, uint32_t* flags) {
  const int64_t quads = (int64_t)S * rows * K / 4;
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= quads) return;
  const int64_t flat = q * 4;                 // index into [S][rows][K]
  const int j = (int)(flat % K);
  const int64_t sr = flat / K;
  const int r = (int)(sr % rows), s = (int)(sr / rows);
  const int4 li = *reinterpret_cast<const int4*>(local_idx + flat);
  const float* row = logits + ((int64_t)s * rows + r) * ld;
  const int l4[4] = {li.x, li.y, li.z, li.w};
  float2 o[4];
  bool bad = false;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int l = l4[u];
    if (l >= 0 && l < ld) {
      o[u] = make_float2(__ldg(row + l), __int_as_float((int)global_of(s, l, S, I)));
    } else {
      bad |= l >= ld;
      o[u] = make_float2(-INFINITY, __int_as_float(-1));
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);
  float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float2*>(cand) + ((int64_t)r * S + s) * K + j);
  dst[0] = make_float4(o[0].x, o[0].y, o[1].x, o[1].y);
  dst[1] = make_float4(o[2].x, o[2].y, o[3].x, o[3].y);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status check_common(const float* logits, int64_t ld, int rows, int S, int I, int K) {
  if (!logits || rows < 0 || ld < 4 || (ld & 3) || !aligned16(logits)) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (ld > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)rows * S > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

template <bool kPack>
dsa_status launch_topk(const float* logits, int64_t ld, int rows, int S, int I, int K,
                       const int32_t* row_starts, const int32_t* row_ends, int32_t* local_idx,
                       float* cand, uint32_t* err_flags, cudaStream_t stream) {
  const int stage_cap = ld < kStageCapElems ? (int)ld : kStageCapElems;
  const size_t smem = topk_stage_offset() + (size_t)stage_cap * sizeof(float);
  auto kern = shard_topk_kernel<kPack>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  kern<<<rows * S, kTopkThreads, smem, stream>>>(logits, ld, rows, S, I, K, row_starts, row_ends,
                                                 local_idx, cand, err_flags, stage_cap);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_shard_topk(const float* logits, int64_t ld, int rows, int S, int I,
                                     int K, const int32_t* row_starts, const int32_t* row_ends,
                                     int32_t* local_idx, uint32_t* err_flags,
                                     cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (!row_ends || !local_idx) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  return launch_topk<false>(logits, ld, rows, S, I, K, row_starts, row_ends, local_idx, nullptr,
                            err_flags, stream);
}

extern "C" dsa_status dsa_shard_topk_pack(const float* logits, int64_t ld, int rows, int S,
                                          int I, int K, const int32_t* row_starts,
                                          const int32_t* row_ends, int32_t* local_idx,
                                          float* cand, uint32_t* err_flags,
                                          cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (!row_ends || !cand || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  return launch_topk<true>(logits, ld, rows, S, I, K, row_starts, row_ends, local_idx, cand,
                           err_flags, stream);
}

extern "C" dsa_status dsa_pack_candidates(const float* logits, int64_t ld,
                                          const int32_t* local_idx, int rows, int S, int I,
                                          int K, float* cand, uint32_t* err_flags,
                                          cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (!local_idx || !cand || !aligned16(local_idx) || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  const int64_t quads = (int64_t)S * rows * K / 4;
  const int64_t blocks = (quads + 255) / 256;
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(logits, ld, local_idx, rows, S, I, K, cand,
                                                    err_flags);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
