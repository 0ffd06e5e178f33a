// The PCP prefill path's cache rows (sm_103a): RMS norm of the latent kv_c
// and interleaved rotation of k_pe for each new token, the rows materialised
// for the gather across PCP ranks and/or written into the paged KV cache, and
// the insert of gathered rows (PR #52046 report, "DSV3.2 PCP sharding",
// sections 功能与动机, 实现拆解 items 1 and 3 and 关键源码片段:
// `_fused_norm_rope_kernel` pid == 1, `maybe_gather_mla_latent_cache_inputs`,
// `do_kv_cache_update`).
//
// One warp per token.  kv_c (512 bf16 = 1 KB) is 32 bytes a lane (two
// 16-byte loads), its sum of squares a warp reduction; k_pe (64 bf16) is one
// rotation pair a lane.  A cache row is kv_c then the rotated k_pe (576 bf16,
// 1152 bytes): every lane writes 32 bytes of the first part and 4 of the
// second, so each token's stores are whole 32-byte sectors.  Both kernels are
// bound by HBM bandwidth.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kDc = DSA_MLA_DV;                // 512
constexpr int kDr = DSA_MLA_DQK - DSA_MLA_DV;  // 64
constexpr int kWarps = 8;

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t f32_to_bf16(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__global__ void __launch_bounds__(kWarps * 32)
    fused_norm_rope_kernel(const uint16_t* __restrict__ kv_c, const uint16_t* __restrict__ k_pe,
                           const int32_t* __restrict__ positions,
                           const float* __restrict__ weight, float eps,
                           const float* __restrict__ cos_sin, int max_pos, int T,
                           uint16_t* __restrict__ kv_out, uint16_t* __restrict__ kpe_out,
                           const int32_t* __restrict__ slot_mapping,
                           uint16_t* __restrict__ kv_cache, int64_t n_slots, uint32_t* flags) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;

  // kv_c: elements 16 lane .. 16 lane + 15.
  const uint4* src = reinterpret_cast<const uint4*>(kv_c + (int64_t)t * kDc) + 2 * lane;
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_to_f32(wd[i] & 0xFFFFu);
    x[2 * i + 1] = bf16_to_f32(wd[i] >> 16);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
  const float inv = rsqrtf(ss * (1.0f / kDc) + eps);
  const float4* w4 = reinterpret_cast<const float4*>(weight) + 4 * lane;
  uint32_t y[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 ww = __ldg(w4 + i);
    y[2 * i] = f32_to_bf16(x[4 * i] * inv * ww.x) | (f32_to_bf16(x[4 * i + 1] * inv * ww.y) << 16);
    y[2 * i + 1] =
        f32_to_bf16(x[4 * i + 2] * inv * ww.z) | (f32_to_bf16(x[4 * i + 3] * inv * ww.w) << 16);
  }

  // k_pe: the lane's pair (2 lane, 2 lane + 1), rotated by the table's angle
  // `lane` of the token's position (cos in the first half, sin in the second).
  const uint32_t pair = __ldg(reinterpret_cast<const uint32_t*>(k_pe + (int64_t)t * kDr) + lane);
  const int pos = positions[t];
  float c = 1.f, s = 0.f;
  if (pos >= 0 && pos < max_pos) {
    c = __ldg(cos_sin + (int64_t)pos * kDr + lane);
    s = __ldg(cos_sin + (int64_t)pos * kDr + kDr / 2 + lane);
  } else if (lane == 0) {
    raise_flag(flags, DSA_FLAG_BOUNDS);   // identity rotation for this token
  }
  const float x1 = bf16_to_f32(pair & 0xFFFFu), x2 = bf16_to_f32(pair >> 16);
  const uint32_t r = f32_to_bf16(fmaf(x1, c, -x2 * s)) | (f32_to_bf16(fmaf(x2, c, x1 * s)) << 16);

  const uint4 y0 = make_uint4(y[0], y[1], y[2], y[3]), y1 = make_uint4(y[4], y[5], y[6], y[7]);
  if (kv_out) {
    uint4* dst = reinterpret_cast<uint4*>(kv_out + (int64_t)t * kDc) + 2 * lane;
    dst[0] = y0;
    dst[1] = y1;
    reinterpret_cast<uint32_t*>(kpe_out + (int64_t)t * kDr)[lane] = r;
  }
  if (slot_mapping) {
    const int64_t slot = slot_mapping[t];
    if (slot >= n_slots) {
      if (lane == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
    } else if (slot >= 0) {
      uint16_t* row = kv_cache + slot * (kDc + kDr);
      uint4* dst = reinterpret_cast<uint4*>(row) + 2 * lane;
      dst[0] = y0;
      dst[1] = y1;
      reinterpret_cast<uint32_t*>(row + kDc)[lane] = r;
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    cache_insert_kernel(const uint16_t* __restrict__ kv_rows,
                        const uint16_t* __restrict__ kpe_rows,
                        const int32_t* __restrict__ slot_mapping, int T,
                        uint16_t* __restrict__ kv_cache, int64_t n_slots, uint32_t* flags) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= n_slots) {
    if (lane == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(kv_rows + (int64_t)t * kDc) + 2 * lane;
  const uint4 a = __ldg(src), b = __ldg(src + 1);
  const uint32_t r = __ldg(reinterpret_cast<const uint32_t*>(kpe_rows + (int64_t)t * kDr) + lane);
  uint16_t* row = kv_cache + slot * (kDc + kDr);
  uint4* dst = reinterpret_cast<uint4*>(row) + 2 * lane;
  dst[0] = a;
  dst[1] = b;
  reinterpret_cast<uint32_t*>(row + kDc)[lane] = r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_fused_norm_rope(const uint16_t* kv_c, const uint16_t* k_pe,
                                          const int32_t* positions, const float* norm_weight,
                                          float eps, const float* cos_sin_cache, int max_pos,
                                          int T, uint16_t* kv_out, uint16_t* kpe_out,
                                          const int32_t* slot_mapping, uint16_t* kv_cache,
                                          int64_t n_slots, uint32_t* err_flags,
                                          cudaStream_t stream) {
  if (T < 0 || max_pos < 1 || !(eps >= 0.f) || !std::isfinite(eps)) return DSA_ERR_INVALID_ARG;
  if ((kv_out == nullptr) != (kpe_out == nullptr) ||
      (slot_mapping == nullptr) != (kv_cache == nullptr))
    return DSA_ERR_INVALID_ARG;
  if (!kv_out && !slot_mapping) return DSA_ERR_INVALID_ARG;   // nothing to produce
  if (slot_mapping && n_slots < 1) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (!kv_c || !k_pe || !positions || !norm_weight || !cos_sin_cache) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv_c) || !aligned16(norm_weight) || (reinterpret_cast<uintptr_t>(k_pe) & 3u) ||
      (kv_out && (!aligned16(kv_out) || (reinterpret_cast<uintptr_t>(kpe_out) & 3u))) ||
      (kv_cache && !aligned16(kv_cache)))
    return DSA_ERR_INVALID_ARG;
  const unsigned grid = (unsigned)((T + kWarps - 1) / kWarps);
  const cudaError_t e = launch_kernel(fused_norm_rope_kernel, dim3(grid), dim3(kWarps * 32), 0,
                                      stream, 0, kv_c, k_pe, positions, norm_weight, eps,
                                      cos_sin_cache, max_pos, T, kv_out, kpe_out, slot_mapping,
                                      kv_cache, n_slots, err_flags);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" dsa_status dsa_kv_cache_insert(const uint16_t* kv_rows, const uint16_t* kpe_rows,
                                          const int32_t* slot_mapping, int T,
                                          uint16_t* kv_cache, int64_t n_slots,
                                          uint32_t* err_flags, cudaStream_t stream) {
  if (T < 0 || n_slots < 1) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (!kv_rows || !kpe_rows || !slot_mapping || !kv_cache) return DSA_ERR_INVALID_ARG;
  if (!aligned16(kv_rows) || (reinterpret_cast<uintptr_t>(kpe_rows) & 3u) || !aligned16(kv_cache))
    return DSA_ERR_INVALID_ARG;
  const unsigned grid = (unsigned)((T + kWarps - 1) / kWarps);
  const cudaError_t e = launch_kernel(cache_insert_kernel, dim3(grid), dim3(kWarps * 32), 0,
                                      stream, 0, kv_rows, kpe_rows, slot_mapping, T, kv_cache,
                                      n_slots, err_flags);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
