// Device helpers shared by the DCP sparse-indexer kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "dsa.h"
#include "fastdiv.h"

namespace dsa {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Order-preserving keys.
//
// score_key maps an fp32 score to a uint32 whose unsigned order is the score
// order (NaN excluded); -0.0 is folded into +0.0 so the two tie.  Ties on the
// score are broken toward the smaller global token id, so a candidate's full
// rank key is (score_key << 32) | ~id: larger key = better candidate.  A valid
// score never maps below 0x007FFFFF (the key of -inf), so the 64-bit key 0 is
// free to mean "padding".
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t score_key(float f) {
  // f + 0 turns -0.0 into +0.0 (round to nearest, no flush of denormals);
  // then negative patterns are inverted and positive ones get the top bit:
  // b ^ (sign-extended sign | 0x80000000).
  const uint32_t b = __float_as_uint(__fadd_rn(f, 0.0f));
  return b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ---------------------------------------------------------------------------
// Interleaved DCP sharding, closed forms of the ownership rule
// owner(t) = (t / I) mod S (PR #46076 report, "[Attention][DSA] support dcp for
// FLASHINFER_MLA_SPARSE", section 关键源码片段, `_dcp_localize_decode_seq_lens`).
// A shard keeps its tokens in increasing global order: token t is local slot
// (t / (I S)) I + t mod I of shard (t / I) mod S, and local slot l of shard s
// is token (l / I) I S + s I + l mod I.  The maps work on 32-bit ids (row
// ends are int32), with the divisions by I, I*S and S precomputed on the host
// (fastdiv.h).
// ---------------------------------------------------------------------------
struct ShardMath {
  int S, I;
  FastDiv fI, fIS, fS;
  ShardMath() : S(1), I(1) {}
  ShardMath(int S_, int I_) : S(S_), I(I_), fI(I_), fIS((uint32_t)(I_ * S_)), fS(S_) {}

  __device__ __forceinline__ int owner(uint32_t t) const {
    const uint32_t q = fdiv(t, fI);
    return (int)(q - fdiv(q, fS) * (uint32_t)S);
  }
  __device__ __forceinline__ uint32_t local_slot(uint32_t t) const {
    uint32_t r;
    fdivmod(t, fI, &r);
    return fdiv(t, fIS) * (uint32_t)I + r;
  }
  __device__ __forceinline__ uint32_t global_id(int s, uint32_t l) const {
    uint32_t r;
    const uint32_t q = fdivmod(l, fI, &r);
    return q * fIS.d + (uint32_t)s * (uint32_t)I + r;
  }
  // Tokens of the global prefix [0, L) that shard s holds (L < 2^31).
  __device__ __forceinline__ uint32_t local_len(uint32_t L, int s) const {
    uint32_t r;
    const uint32_t q = fdivmod(L, fIS, &r);
    const int rem = min(max((int)r - s * I, 0), I);
    return q * (uint32_t)I + (uint32_t)rem;
  }
};

// 4-byte asynchronous copy global -> shared (cp.async); completion is waited
// for by cp_async_wait_all, after which a barrier makes it visible to the CTA.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void raise_flag(uint32_t* flags, uint32_t bit) {
  if (flags) atomicOr(flags, bit);
}

// ---------------------------------------------------------------------------
// Bulk async copies (TMA, non-tensor form) global -> shared, completed on an
// mbarrier.  Both addresses 16-byte aligned, size a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false (and the
// caller raises DSA_FLAG_TIMEOUT) after `limit` polls; each poll may suspend
// the thread for a hardware-chosen interval, so the bound is generous.
#ifdef DSA_TEST_STALLED_COPY
constexpr uint32_t kWaitPolls = 1u << 12;   // the test build's short bound
#else
constexpr uint32_t kWaitPolls = 1u << 22;
#endif
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

// ---------------------------------------------------------------------------
// Block-wide exclusive prefix sum of one int per thread.  `scratch` holds at
// least blockDim.x/32 + 1 ints.  Returns the exclusive prefix; *total gets the
// sum over the block.  Contains two __syncthreads().
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
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
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
    int incl = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nwarps) scratch[lane] = incl - w;
    if (lane == 31) scratch[32] = incl;
  }
  __syncthreads();
  *total = scratch[32];
  return scratch[warp] + x - v;
}

// Host: launch `kernel` on `stream`, in clusters of cluster_x CTAs along x when
// cluster_x > 0.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int n = 0;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace dsa
