// LSE combine of the shards' partial attention outputs.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 实现拆解 item 5 and section 评论区精华 (LSE base normalisation: the
// sparse MLA kernel reports a base-2 LSE, the DCP reducer needs base e);
// PR #52046 report, "DSV3.2 PCP sharding", section 关键源码片段
// (`dcp_manager.combine` of attn_out by lse).
//
// Per (row, head): lambda_s = lse2_s ln 2, M = max lambda_s,
// w_s = exp(lambda_s - M), out = sum w_s O_s / sum w_s, lse = M + ln sum w_s.
// Since exp((lse2_s - max lse2) ln 2) = 2^(lse2_s - max lse2) exactly, the
// weights are taken with exp2 on the base-2 values and only the final LSE is
// converted; that is the same quantity with one rounding fewer per weight.
//
// Up to 8 shards: one warp per (row, head, 256-wide slice of D), every shard's
// 16-byte load in flight at once.  More shards: one warp per (row, head), each
// lane streaming 8 bf16 per shard per slice; shards whose LSE is -inf are not
// read.
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kCombThreads = 256;
constexpr int kCombWarps = kCombThreads / 32;
constexpr float kLn2 = 0.693147180559945309417f;

__device__ __forceinline__ void accum8(float* acc, uint4 v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    acc[2 * q] = fmaf(w, __uint_as_float(u[q] << 16), acc[2 * q]);
    acc[2 * q + 1] = fmaf(w, __uint_as_float(u[q] & 0xffff0000u), acc[2 * q + 1]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kCombThreads)
    lse_combine_kernel(const uint16_t* __restrict__ part, const float* __restrict__ lse2,
                       int S, int rows, int H, int D, uint16_t* __restrict__ out,
                       float* __restrict__ lse_out) {
  const int64_t rh = (int64_t)blockIdx.x * kCombWarps + (threadIdx.x >> 5);
  const int64_t RH = (int64_t)rows * H;
  if (rh >= RH) return;
  const int lane = threadIdx.x & 31;

  const float a0 = lane < S ? __ldg(lse2 + lane * RH + rh) : -INFINITY;
  const float a1 = lane + 32 < S ? __ldg(lse2 + (lane + 32) * RH + rh) : -INFINITY;
  float M = fmaxf(a0, a1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  uint16_t* dst = out + rh * D;
  if (M == -INFINITY) {  // no shard holds anything
    for (int d = lane * 8; d < D; d += 256)
      *reinterpret_cast<uint4*>(dst + d) = make_uint4(0u, 0u, 0u, 0u);
    if (lse_out && lane == 0) lse_out[rh] = -INFINITY;
    return;
  }
  // The slice loop below is warp-uniform (the shuffles need every lane); a
  // lane past the end of D only skips its loads and its store.
  const float w0 = a0 == -INFINITY ? 0.f : exp2f(a0 - M);
  const float w1 = a1 == -INFINITY ? 0.f : exp2f(a1 - M);
  float wsum = w0 + w1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(kFull, wsum, o);
  const float inv = 1.f / wsum;

  for (int d0 = 0; d0 < D; d0 += 256) {
    const int d = d0 + lane * 8;
    const bool in = d < D;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 4) {
      uint4 v[4];
      float w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = s0 + u;
        const float ws = __shfl_sync(kFull, s < 32 ? w0 : w1, s & 31);
        w[u] = s < S ? ws : 0.f;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (in && w[u] != 0.f)
          v[u] = __ldg(reinterpret_cast<const uint4*>(part + ((int64_t)s * RH + rh) * D + d));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (w[u] != 0.f) accum8(acc, v[u], w[u]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    if (in) *reinterpret_cast<uint4*>(dst + d) = o;
  }
  if (lse_out && lane == 0) lse_out[rh] = (M + log2f(wsum)) * kLn2;
}

// Up to 8 shards: a persistent grid; each warp walks (row, head, 256-element
// slice of D) items and, while it combines one item, already has the next
// item's loads in flight (every shard's 16-byte load per lane, issued
// unconditionally: an empty shard's values are loaded but not used, and its
// LSE).  SN >= S shards are held in registers.
// Resident blocks per SM: fewer when each warp holds more shards in flight, so
// the double-buffered loads stay in registers.
template <int SN>
constexpr int persist_blocks() { return SN <= 4 ? 4 : 2; }

// Item -> (row * H + head, 256-element slice).  Below 2^31 items (k32) the
// division by the slice count uses its host-computed invariant divisor.
template <bool k32>
__device__ __forceinline__ int64_t split_item(int64_t item, int nsl, const FastDiv& fnsl,
                                              int* sl) {
  if (k32) {
    uint32_t r;
    const uint32_t q = fdivmod((uint32_t)item, fnsl, &r);
    *sl = (int)r;
    return q;
  }
  const int64_t rh = item / nsl;
  *sl = (int)(item - rh * nsl);
  return rh;
}

template <int SN, bool k32>
__device__ __forceinline__ void load_item(const uint16_t* __restrict__ part,
                                          const float* __restrict__ lse2, int S, int64_t RH,
                                          int D, int nsl, const FastDiv& fnsl, int64_t item,
                                          uint4 (&v)[SN], float& a) {
  const int lane = threadIdx.x & 31;
  int sl;
  const int64_t rh = split_item<k32>(item, nsl, fnsl, &sl);
  const int d = sl * 256 + lane * 8;
#pragma unroll
  for (int s = 0; s < SN; ++s)
    v[s] = (s < S && d < D)
               ? __ldg(reinterpret_cast<const uint4*>(part + ((int64_t)s * RH + rh) * D + d))
               : make_uint4(0u, 0u, 0u, 0u);
  a = lane < S ? __ldg(lse2 + lane * RH + rh) : -INFINITY;
}

template <int SN, bool k32>
__global__ void __launch_bounds__(kCombThreads, persist_blocks<SN>())
    lse_combine_persist_kernel(const uint16_t* __restrict__ part, const float* __restrict__ lse2,
                               int S, int rows, int H, int D, uint16_t* __restrict__ out,
                               float* __restrict__ lse_out, const FastDiv fnsl) {
  const int nsl = (D + 255) >> 8;
  const int64_t RH = (int64_t)rows * H;
  const int64_t nitems = RH * nsl;
  const int64_t stride = (int64_t)gridDim.x * kCombWarps;
  const int lane = threadIdx.x & 31;
  int64_t item = (int64_t)blockIdx.x * kCombWarps + (threadIdx.x >> 5);
  uint4 cur[SN], nxt[SN];
  float a_cur = -INFINITY, a_nxt = -INFINITY;
  if (item < nitems) load_item<SN, k32>(part, lse2, S, RH, D, nsl, fnsl, item, cur, a_cur);
  for (; item < nitems; item += stride) {
    const int64_t next = item + stride;
    if (next < nitems) load_item<SN, k32>(part, lse2, S, RH, D, nsl, fnsl, next, nxt, a_nxt);
    int sl;
    const int64_t rh = split_item<k32>(item, nsl, fnsl, &sl);
    const int d = sl * 256 + lane * 8;
    uint16_t* dst = out + rh * D;
    float M = a_cur;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (M == -INFINITY) {  // no shard holds anything
      if (d < D) *reinterpret_cast<uint4*>(dst + d) = make_uint4(0u, 0u, 0u, 0u);
      if (lse_out && sl == 0 && lane == 0) lse_out[rh] = -INFINITY;
    } else {
      const float w0 = a_cur == -INFINITY ? 0.f : exp2f(a_cur - M);
      float wsum = w0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(kFull, wsum, o);
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
      for (int s = 0; s < SN; ++s) {
        const float ws = __shfl_sync(kFull, w0, s);
        if (s < S && ws != 0.f) accum8(acc, cur[s], ws);
      }
      const float inv = 1.f / wsum;
      if (d < D) {
        uint4 o;
        o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(dst + d) = o;
      }
      if (lse_out && sl == 0 && lane == 0) lse_out[rh] = (M + log2f(wsum)) * kLn2;
    }
#pragma unroll
    for (int s = 0; s < SN; ++s) cur[s] = nxt[s];
    a_cur = a_nxt;
  }
}

template <int SN>
dsa_status launch_persist(const uint16_t* part, const float* lse2, int S, int rows, int H, int D,
                          uint16_t* out, float* lse_out, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  const int64_t items = (int64_t)rows * H * ((D + 255) / 256);
  const int64_t need = (items + kCombWarps - 1) / kCombWarps;
  const int64_t cap = (int64_t)sms * persist_blocks<SN>();
  const int blocks = (int)(need < cap ? need : cap);
  const int nsl = (D + 255) / 256;
  // 32-bit items when every item index (and the index one stride past the
  // last) stays below 2^31.
  const bool k32 = items + (int64_t)blocks * kCombWarps < ((int64_t)1 << 31);
  auto kern = k32 ? lse_combine_persist_kernel<SN, true> : lse_combine_persist_kernel<SN, false>;
  const cudaError_t e = launch_kernel(kern, dim3((unsigned)blocks), dim3(kCombThreads), 0, stream,
                                      0, part, lse2, S, rows, H, D, out, lse_out,
                                      FastDiv((uint32_t)nsl));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_lse_combine(const uint16_t* partial_out, const float* lse2, int S,
                                      int rows, int H, int D, uint16_t* out, float* lse_out,
                                      uint32_t* err_flags, cudaStream_t stream) {
  (void)err_flags;   // no asynchronous copies on this path: nothing can stall
  if (rows < 0 || H < 1 || D < 8 || (D & 7)) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!partial_out || !lse2 || !out || !aligned16(partial_out) || !aligned16(out))
    return DSA_ERR_INVALID_ARG;
  if (S <= 2) return launch_persist<2>(partial_out, lse2, S, rows, H, D, out, lse_out, stream);
  if (S <= 4) return launch_persist<4>(partial_out, lse2, S, rows, H, D, out, lse_out, stream);
  if (S <= 8) return launch_persist<8>(partial_out, lse2, S, rows, H, D, out, lse_out, stream);
  {
    const int64_t warps = (int64_t)rows * H;
    const int64_t blocks = (warps + kCombWarps - 1) / kCombWarps;
    if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
    const cudaError_t e = launch_kernel(lse_combine_kernel, dim3((unsigned)blocks),
                                        dim3(kCombThreads), 0, stream, 0, partial_out, lse2, S,
                                        rows, H, D, out, lse_out);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
}
