// Sparse MLA decode attention of every shard over its compacted KV slots.
//
// PR #52046 report, "DSV3.2 PCP sharding", section 关键源码片段:
// `_fused_norm_rope_kernel` writes a cache row as the normed latent kv_c
// followed by the roped k_pe; `_sparse_indexer_and_attn` concatenates the MQA
// query's parts on the last dimension and `forward_mqa(q, kv_cache, ...)`
// returns each shard's output and LSE for `dcp_manager.combine`.  PR #46076
// report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE", section
// 实现拆解 items 4 and 5: the kernel reads the compacted slots and returns a
// base-2 LSE.
//
// Per (shard s, row r, head h): s_j = scale * (q[r][h] . row_j) over the
// shard's slots[s][r][0 .. counts[s][r]), O = sum_j 2^(s_j log2 e) v_j /
// sum_j 2^(s_j log2 e) with v_j the first 512 entries of row_j, and
// lse2 = log2 sum_j exp(s_j).
//
// One CTA per (row, shard, group of 64 heads), tensor cores through mma.sync
// m16n8k16 (bf16 in, fp32 accumulate), warp-specialised:
//  * a producer warp gathers the shard's selected cache rows by slot, one row
//    per lane and one bulk asynchronous copy (TMA, non-tensor form) per row,
//    into two stages of 32 tokens guarded by full / empty mbarriers (invalid
//    tokens are zeroed and masked);
//  * eight consumer warps, a pair per 16 heads: each warp of a pair computes
//    the scores of its 16 heads against half of the tile's tokens (all 576
//    dimensions), the pair swaps them through shared memory under one
//    64-thread named barrier, and each warp then runs the online softmax (exp2
//    domain) on all 32 tokens and O += P V for its half of the 512 output
//    dimensions (128 fp32 accumulators per thread); the softmax weights go
//    from the score registers straight into the operand layout of P V.
// No block-wide barrier runs inside the token loop; every wait is bounded.
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kDqk = DSA_MLA_DQK;            // 576: latent 512 + rope 64
constexpr int kDv = DSA_MLA_DV;              // 512
constexpr int kHeads = 64;                   // heads per CTA: four blocks of 16
constexpr int kHalfDv = kDv / 2;             // output dimensions per consumer warp
constexpr int kTile = 32;                    // tokens per stage (one per producer lane)
constexpr int kStages = 2;
constexpr int kConsumers = 8;                // warps 0..7; warp 8 produces
constexpr int kAttnThreads = (kConsumers + 1) * 32;
constexpr int kStride = kDqk + 8;            // smem row stride (elements): rows 16 B apart in banks
constexpr int kChunks = kDqk / 8;            // 16-byte chunks per row
constexpr uint32_t kRowBytes = kDqk * 2;     // one cache row, one bulk copy
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kDqk % 32 == 0 && kHalfDv % 16 == 0, "tile shapes");
static_assert(kTile == 32 && kStages == 2, "one token per producer lane; parity = tile & 1");

struct AttnSmem {
  uint64_t full[kStages];                    // a stage's rows have landed
  uint64_t empty[kStages];                   // every consumer warp is done with a stage
  alignas(16) __nv_bfloat16 q[kHeads * kStride];
  alignas(16) __nv_bfloat16 kv[kStages][kTile * kStride];
  // Score swap between the two warps of a head block: [block][token half]
  // [tile parity][value][lane], each lane's eight scores of its half.
  float xs[kHeads / 16][2][2][8][32];
  uint32_t vmask[kStages];                   // bit i: token i of the stage is valid
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Named barrier over `count` threads that also returns whether any of them
// passed pred = true.
__device__ __forceinline__ bool bar_any(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

struct AttnArgs {
  const __nv_bfloat16* q;        // [rows][H][kDqk]
  const __nv_bfloat16* cache;    // [S][n_slots][kDqk]
  int64_t n_slots;
  const int32_t* slots;          // [S][rows][K]
  const int32_t* counts;         // [S][rows]
  int rows, S, H, K;
  float c2;                      // scale * log2(e)
  __nv_bfloat16* out;            // [S][rows][H][kDv]
  float* lse2;                   // [S][rows][H]
  uint32_t* flags;
};

// Producer warp: tile t of 32 tokens into stage t & 1, lane i taking token i.
__device__ __forceinline__ void produce(const AttnArgs& a, AttnSmem& sm, int count, int ntiles,
                                        const int32_t* slot_row,
                                        const __nv_bfloat16* shard_cache) {
  const int lane = threadIdx.x & 31;
  bool bad = false, ok = true;
  int issued = 0;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    if (t >= kStages) ok = mbar_wait(&sm.empty[st], (uint32_t)(t / kStages - 1) & 1u);
    if (!__all_sync(kFull, ok)) {
      ok = false;
      break;
    }
    const int idx = t * kTile + lane;
    const int slot = idx < count ? __ldg(slot_row + idx) : -1;
    const bool in = slot >= 0 && (int64_t)slot < a.n_slots;
    bad |= idx < count && !in;
    __nv_bfloat16* dst = &sm.kv[st][lane * kStride];
    if (!in)
      for (int c = 0; c < kChunks; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
    const unsigned valid = __ballot_sync(kFull, in);
    if (lane == 0) sm.vmask[st] = valid;
    // The consumers' reads of this stage (generic proxy) before the copies.
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    // Arm first (zeroed rows and flags published by this arrival), then copy.
    if (lane == 0) mbar_expect_tx(&sm.full[st], (uint32_t)__popc(valid) * kRowBytes);
    __syncwarp();
    if (in) bulk_g2s(dst, shard_cache + (int64_t)slot * kDqk, kRowBytes, &sm.full[st]);
    issued = t + 1;
  }
  if (!ok && lane == 0) raise_flag(a.flags, DSA_FLAG_TIMEOUT);
  if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  // Copies still in flight land before this warp, and so the block, exits.
  for (int t = max(0, issued - kStages); t < issued; ++t)
    mbar_wait(&sm.full[t & 1], (uint32_t)(t / kStages) & 1u);
}

__global__ void __launch_bounds__(kAttnThreads, 1) sparse_mla_decode_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) unsigned char attn_smem[];
  AttnSmem& sm = *reinterpret_cast<AttnSmem*>(attn_smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int hgroups = a.H / kHeads;
  const int hg = blockIdx.x % hgroups;
  const int pair = blockIdx.x / hgroups;     // s * rows + r
  const int s = pair / a.rows, r = pair - s * a.rows;
  int count = __ldg(a.counts + pair);
  if ((count < 0 || count > a.K) && tid == 0) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  count = min(max(count, 0), a.K);
  const int64_t obase = (int64_t)pair * a.H + hg * kHeads;   // first head of the group

  if (count == 0) {
    // Nothing selected on this shard: O = 0, lse2 = -inf.
    for (int i = tid; i < kHeads * kDv / 8; i += kAttnThreads)
      *reinterpret_cast<uint4*>(a.out + (obase + i / (kDv / 8)) * kDv + (i % (kDv / 8)) * 8) =
          make_uint4(0, 0, 0, 0);
    if (tid < kHeads) a.lse2[obase + tid] = -INFINITY;
    return;
  }

  // The group's query rows (cp.async by every thread) and the barriers.
  {
    const __nv_bfloat16* qg = a.q + ((int64_t)r * a.H + hg * kHeads) * kDqk;
    for (int c = tid; c < kHeads * kChunks; c += kAttnThreads) {
      const int h = c / kChunks, j = c - h * kChunks;
      cp_async16(&sm.q[h * kStride + j * 8], qg + (int64_t)h * kDqk + j * 8);
    }
    cp_async_commit();
  }
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kConsumers);
    }
    mbar_init_fence();
  }
  cp_async_wait_all();
  __syncthreads();
  const int ntiles = (count + kTile - 1) / kTile;

  if (warp == kConsumers) {
    produce(a, sm, count, ntiles, a.slots + (int64_t)pair * a.K,
            a.cache + (int64_t)s * a.n_slots * kDqk);
    return;
  }

  // ---- consumer warps: head block hb (16 heads), half dh -------------------
  const int hb = warp >> 1, dh = warp & 1;
  const uint32_t qa = smem_u32(&sm.q[(hb * 16 + (lane & 15)) * kStride + (lane >> 4) * 8]);
  float acc[kHalfDv / 8][4];                 // 32 n-tiles of 8 dims x (rows g, g + 8)
#pragma unroll
  for (int j = 0; j < kHalfDv / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  // Running max and two row sums: of the fp32 weights (for the LSE) and of
  // the bf16-rounded weights that enter P V (to normalise O, which is then an
  // exact convex mix of what was multiplied).
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, w0 = 0.f, w1 = 0.f;
  bool ok = true;

  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    const bool landed = mbar_wait(&sm.full[st], (uint32_t)(t / kStages) & 1u);

    // Scores of the 16 heads against tokens dh*16 .. dh*16+15 (two n-tiles),
    // even and odd k-steps in separate accumulators.
    float c[2][2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 2; ++e) c[n][e][0] = c[n][e][1] = c[n][e][2] = c[n][e][3] = 0.f;
    const uint32_t kb = smem_u32(&sm.kv[st][(dh * 16 + (lane & 7) + ((lane >> 4) & 1) * 8) *
                                                kStride + ((lane >> 3) & 1) * 8]);
#pragma unroll 3
    for (int ks = 0; ks < kDqk / 16; ks += 2) {
      uint32_t af[4], bf[4], ag[4], bg[4];
      ldsm_x4(qa + ks * 32, af);
      ldsm_x4(kb + ks * 32, bf);
      ldsm_x4(qa + ks * 32 + 32, ag);
      ldsm_x4(kb + ks * 32 + 32, bg);
      mma_bf16(c[0][0], af, bf[0], bf[1]);
      mma_bf16(c[1][0], af, bf[2], bf[3]);
      mma_bf16(c[0][1], ag, bg[0], bg[1]);
      mma_bf16(c[1][1], ag, bg[2], bg[3]);
    }
    // x[kk][v]: k-step kk (tokens kk*16 ..); v in A-fragment order: rows g
    // (v = 0, 1, 4, 5) and g + 8 (v = 2, 3, 6, 7) at tokens 2t, 2t+1, 2t+8, 2t+9.
    float own[8], oth[8];
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int u = 0; u < 4; ++u) own[4 * n + u] = (c[n][0][u] + c[n][1][u]) * a.c2;
    float* mine = &sm.xs[hb][dh][st][0][lane];
#pragma unroll
    for (int v = 0; v < 8; ++v) mine[v * 32] = own[v];
    if (bar_any(1 + hb, 64, !landed)) {      // both warps of the block see the same answer
      ok = false;
      break;
    }
    const float* other = &sm.xs[hb][dh ^ 1][st][0][lane];
#pragma unroll
    for (int v = 0; v < 8; ++v) oth[v] = other[v * 32];
    float x[2][8];                           // by k-step, selected without indexing by dh
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      x[0][v] = dh ? oth[v] : own[v];
      x[1][v] = dh ? own[v] : oth[v];
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
    const uint32_t vm = sm.vmask[st] >> (2 * t4);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int tok = kk * 16 + (v & 1) + ((v >> 2) << 3);   // + 2 t4, folded into vm
        if (!((vm >> tok) & 1u)) x[kk][v] = -INFINITY;
        if ((v >> 1) & 1) mx1 = fmaxf(mx1, x[kk][v]);
        else mx0 = fmaxf(mx0, x[kk][v]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // Rows with nothing valid yet keep m = -inf: use 0 as the reference.
    const float ref0 = n0 == -INFINITY ? 0.f : n0, ref1 = n1 == -INFINITY ? 0.f : n1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
    m0 = n0;
    m1 = n1;
    uint32_t pa[2][4];
    float s0 = 0.f, s1 = 0.f, r0 = 0.f, r1 = 0.f;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      float e[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) e[v] = exp2f(x[kk][v] - (((v >> 1) & 1) ? ref1 : ref0));
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        pa[kk][q2] = pack_bf16(e[2 * q2], e[2 * q2 + 1]);
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa[kk][q2]));
        if (q2 & 1) {
          s1 += e[2 * q2] + e[2 * q2 + 1];
          r1 += f.x + f.y;
        } else {
          s0 += e[2 * q2] + e[2 * q2 + 1];
          r0 += f.x + f.y;
        }
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      s0 += __shfl_xor_sync(kFull, s0, o);
      s1 += __shfl_xor_sync(kFull, s1, o);
      r0 += __shfl_xor_sync(kFull, r0, o);
      r1 += __shfl_xor_sync(kFull, r1, o);
    }
    l0 = l0 * al0 + s0;
    l1 = l1 * al1 + s1;
    w0 = w0 * al0 + r0;
    w1 = w1 * al1 + r1;
    if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {   // the max moved: rescale O
#pragma unroll
      for (int j = 0; j < kHalfDv / 8; ++j) {
        acc[j][0] *= al0;
        acc[j][1] *= al0;
        acc[j][2] *= al1;
        acc[j][3] *= al1;
      }
    }
    // O += P V over this warp's 256 output dimensions.
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t vb = smem_u32(&sm.kv[st][(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) *
                                                  kStride + dh * kHalfDv + (lane >> 4) * 8]);
#pragma unroll
      for (int j = 0; j < kHalfDv / 16; ++j) {
        uint32_t bf[4];
        ldsm_x4_t(vb + j * 32, bf);
        mma_bf16(acc[2 * j], pa[kk], bf[0], bf[1]);
        mma_bf16(acc[2 * j + 1], pa[kk], bf[2], bf[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[st]);   // this warp is done with the stage
  }
  if (!ok && lane == 0) raise_flag(a.flags, DSA_FLAG_TIMEOUT);

  // ---- O / w in bf16, lse2 = m + log2 l ----------------------------------------
  const float inv0 = w0 > 0.f ? 1.f / w0 : 0.f, inv1 = w1 > 0.f ? 1.f / w1 : 0.f;
  const int64_t h0 = obase + hb * 16 + g;
  __nv_bfloat16* o0 = a.out + h0 * kDv + dh * kHalfDv + 2 * t4;
  __nv_bfloat16* o1 = o0 + 8 * kDv;
#pragma unroll
  for (int j = 0; j < kHalfDv / 8; ++j) {
    *reinterpret_cast<uint32_t*>(o0 + j * 8) = pack_bf16(acc[j][0] * inv0, acc[j][1] * inv0);
    *reinterpret_cast<uint32_t*>(o1 + j * 8) = pack_bf16(acc[j][2] * inv1, acc[j][3] * inv1);
  }
  if (dh == 0 && t4 == 0) {
    a.lse2[h0] = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
    a.lse2[h0 + 8] = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_sparse_mla_decode(const uint16_t* q, const uint16_t* kv_cache,
                                            int64_t n_slots, const int32_t* slots,
                                            const int32_t* counts, int rows, int S, int H, int K,
                                            float scale, uint16_t* out, float* lse2,
                                            uint32_t* err_flags, cudaStream_t stream) {
  if (rows < 0 || K < 1 || n_slots < 1 || !(scale == scale) || isinf(scale))
    return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || H < kHeads || H % kHeads) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!q || !kv_cache || !slots || !counts || !out || !lse2) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  if (n_slots > (int64_t)INT32_MAX + 1) return DSA_ERR_UNSUPPORTED;
  const int64_t blocks = (int64_t)rows * S * (H / kHeads);
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  const int smem = (int)sizeof(AttnSmem);
  if (cudaFuncSetAttribute(sparse_mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const AttnArgs a{reinterpret_cast<const __nv_bfloat16*>(q),
                   reinterpret_cast<const __nv_bfloat16*>(kv_cache),
                   n_slots,
                   slots,
                   counts,
                   rows,
                   S,
                   H,
                   K,
                   scale * kLog2e,
                   reinterpret_cast<__nv_bfloat16*>(out),
                   lse2,
                   err_flags};
  const cudaError_t e = launch_kernel(sparse_mla_decode_kernel, dim3((unsigned)blocks),
                                      dim3(kAttnThreads), (size_t)smem, stream, 0, a);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
