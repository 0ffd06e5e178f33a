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
// order (ties on the score go to the smaller slot, i.e. the smaller global id);
// see local_topk.cuh.
#include "common.cuh"
#include "local_topk.cuh"
#include "reg_topk.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kVec = 8;   // register path: local ranges up to 16384 elements
using RT = RegTopk<kTopkThreads, kVec>;

struct TopkSmem {
  LocalTopkSmem loc;
  RegEmitSmem<kTopkThreads, kVec> es;
  uint32_t list[kListCap];   // keys of the threshold bin
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
                      float* __restrict__ cand, uint32_t* flags, int stage_cap,
                      const ShardMath sh) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  float* stage = reinterpret_cast<float*>(smem_raw + topk_stage_offset());

  const int tid = threadIdx.x;
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

  const int64_t base = lo & ~int64_t(3);
  if (hi - base <= RT::kCap) {
    uint32_t key[kVec][4];
    load_keys<kTopkThreads, kVec>(row, lo, hi, key);
    int eq;
    const SelectResult res = select_regs<kTopkThreads, kVec>(key, K, sm.loc.sel, sm.list, sm.es,
                                                             &eq);
    emit_winners<kTopkThreads, kVec>(key, res.thr, res.take_eq, sm.es,
                                     [&](int p, int e, uint32_t) {
      if (p >= K) return;
      const uint32_t l = (uint32_t)(base + e);
      if (out_idx) out_idx[p] = (int32_t)l;
      if (kPack) out_cand[p] = make_float2(row[l], __int_as_float((int)sh.global_id(s, l)));
    });
    return;
  }
  bool ok;
  const float* data = stage_local_range(row, lo, hi, stage, stage_cap, sm.loc, flags, &ok);
  if (!ok) return;
  local_topk_emit<kTopkThreads>(data, n, K, sm.loc, [&](int p, int i, float v) {
    const uint32_t l = (uint32_t)(lo + i);
    if (out_idx) out_idx[p] = (int32_t)l;
    if (kPack) out_cand[p] = make_float2(v, __int_as_float((int)sh.global_id(s, l)));
  });
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

// Scalar checks first; with rows == 0 nothing is read, so pointers may be NULL.
dsa_status check_common(const float* logits, int64_t ld, int rows, int S, int I, int K) {
  if (rows < 0 || ld < 4 || (ld & 3)) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (ld > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)rows * S > (int64_t)INT32_MAX || (int64_t)I * S > (int64_t)INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (rows > 0 && (!logits || !aligned16(logits))) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

template <bool kPack>
dsa_status launch_topk(const float* logits, int64_t ld, int rows, int S, int I, int K,
                       const int32_t* row_starts, const int32_t* row_ends, int32_t* local_idx,
                       float* cand, uint32_t* err_flags, cudaStream_t stream) {
  // Rows that fit the register path need no staging area.
  const int stage_cap = ld <= RT::kCap ? 0 : (ld < kStageCapElems ? (int)ld : kStageCapElems);
  const size_t smem = topk_stage_offset() + (size_t)stage_cap * sizeof(float);
  auto kern = shard_topk_kernel<kPack>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  const cudaError_t e = launch_kernel(kern, dim3((unsigned)(rows * S)), dim3(kTopkThreads), smem,
                                      stream, 0, logits, ld, rows, S, I, K, row_starts, row_ends,
                                      local_idx, cand, err_flags, stage_cap, ShardMath(S, I));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
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
  if (rows == 0) return DSA_OK;
  if (!row_ends || !local_idx) return DSA_ERR_INVALID_ARG;
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
  if (rows == 0) return DSA_OK;
  if (!row_ends || !cand || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  return launch_topk<true>(logits, ld, rows, S, I, K, row_starts, row_ends, local_idx, cand,
                           err_flags, stream);
}

extern "C" dsa_status dsa_pack_candidates(const float* logits, int64_t ld,
                                          const int32_t* local_idx, int rows, int S, int I,
                                          int K, float* cand, uint32_t* err_flags,
                                          cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (rows == 0) return DSA_OK;
  if (!local_idx || !cand || !aligned16(local_idx) || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  const int64_t quads = (int64_t)S * rows * K / 4;
  const int64_t blocks = (quads + 255) / 256;
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  const cudaError_t e = launch_kernel(pack_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 0,
                                      logits, ld, local_idx, rows, S, I, K, cand, err_flags);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
