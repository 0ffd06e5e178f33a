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
// One CTA per (row, shard, group of 32 heads), 8 warps, tensor cores through
// mma.sync m16n8k16 (bf16 in, fp32 accumulate).  The group's 32 query rows
// sit in shared memory; the selected cache rows are gathered by slot into
// double-buffered tiles of 16 tokens with cp.async (invalid tokens are
// zero-filled and masked).  Per tile: the 32 x 16 scores, split over the two
// halves of the 576 dimensions, then an online softmax in the exp2 domain and
// O += P V, each warp owning 16 heads x 128 output dimensions (64 fp32
// accumulators per thread).
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kDqk = DSA_MLA_DQK;            // 576: latent 512 + rope 64
constexpr int kDv = DSA_MLA_DV;              // 512
constexpr int kHeads = 32;                   // heads per CTA
constexpr int kTile = 16;                    // tokens per tile
constexpr int kAttnThreads = 256;
constexpr int kStride = kDqk + 8;            // smem row stride (elements): rows 16 B apart in banks
constexpr int kChunks = kDqk / 8;            // 16-byte chunks per row
constexpr int kKHalf = kDqk / 2;             // 288 dims per score half
constexpr int kSpStride = kTile + 1;
constexpr float kLog2e = 1.4426950408889634f;

static_assert(kDqk % 32 == 0 && kDv % 128 == 0, "tile shapes");

struct AttnSmem {
  alignas(16) __nv_bfloat16 q[kHeads * kStride];
  alignas(16) __nv_bfloat16 kv[2][kTile * kStride];
  float sp[2][kHeads * kSpStride];           // score halves
  int tokv[2][kTile];                        // token valid in this tile
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
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
// 16-byte global -> shared copy; with valid == false the 16 bytes are zero
// filled and nothing is read.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_one() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
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

__global__ void __launch_bounds__(kAttnThreads, 2) sparse_mla_decode_kernel(const AttnArgs a) {
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
  const int32_t* slot_row = a.slots + (int64_t)pair * a.K;
  const __nv_bfloat16* shard_cache = a.cache + (int64_t)s * a.n_slots * kDqk;

  // Warp roles.  Scores: head half hh, token octet nt, dimension half kh.
  // Softmax and P V: head half hh2, output quarter dq.
  const int nt = warp & 1, hh = (warp >> 1) & 1, kh = warp >> 2;
  const int dq = warp & 3, hh2 = warp >> 2;
  const int h_lo = hg * kHeads + hh2 * 16 + g;         // rows g and g + 8 of this warp
  const int64_t obase = (int64_t)pair * a.H;           // (s, r) in [S][rows][H]

  if (count == 0) {
    // Nothing selected on this shard: O = 0, lse2 = -inf.
    for (int i = tid; i < kHeads * kDv / 8; i += kAttnThreads) {
      const int h = hg * kHeads + i / (kDv / 8), c = i % (kDv / 8);
      *reinterpret_cast<uint4*>(a.out + (obase + h) * kDv + c * 8) = make_uint4(0, 0, 0, 0);
    }
    if (tid < kHeads) a.lse2[obase + hg * kHeads + tid] = -INFINITY;
    return;
  }

  // Query rows of the group (their own cp.async group, with the first tile).
  {
    const __nv_bfloat16* qg = a.q + ((int64_t)r * a.H + hg * kHeads) * kDqk;
    for (int c = tid; c < kHeads * kChunks; c += kAttnThreads) {
      const int h = c / kChunks, j = c - h * kChunks;
      cp_async16(&sm.q[h * kStride + j * 8], qg + (int64_t)h * kDqk + j * 8, true);
    }
  }
  const int ntiles = (count + kTile - 1) / kTile;
  bool bad = false;
  auto load_tile = [&](int tile, int buf) {
    for (int c = tid; c < kTile * kChunks; c += kAttnThreads) {
      const int i = c / kChunks, j = c - i * kChunks;
      const int idx = tile * kTile + i;
      int slot = idx < count ? __ldg(slot_row + idx) : -1;
      const bool in = slot >= 0 && (int64_t)slot < a.n_slots;
      bad |= idx < count && !in;
      const __nv_bfloat16* src = in ? shard_cache + (int64_t)slot * kDqk + j * 8 : a.cache;
      cp_async16(&sm.kv[buf][i * kStride + j * 8], src, in);
      if (j == 0) sm.tokv[buf][i] = in;
    }
  };
  load_tile(0, 0);
  cp_async_commit();

  float acc[kDv / 4 / 8][4];                 // 16 n-tiles of 8 dims x (rows g, g + 8)
#pragma unroll
  for (int j = 0; j < kDv / 4 / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  // Running max and two row sums: of the fp32 weights (for the LSE) and of
  // the bf16-rounded weights that enter P V (to normalise O, which is then an
  // exact convex mix of what was multiplied).
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, w0 = 0.f, w1 = 0.f;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int buf = tile & 1;
    __syncthreads();                         // the other buffer and the scores are free
    if (tile + 1 < ntiles) load_tile(tile + 1, buf ^ 1);
    cp_async_commit();                       // possibly empty: keeps the group count uniform
    cp_async_wait_one();                     // this thread's copies of this tile are done
    __syncthreads();                         // ... and everyone's

    // ---- scores: one m16n8 tile per warp over half of the dimensions ------
    {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t qa = smem_u32(&sm.q[(hh * 16 + (lane & 15)) * kStride + kh * kKHalf +
                                         (lane >> 4) * 8]);
      const uint32_t kb = smem_u32(&sm.kv[buf][(nt * 8 + (lane & 7)) * kStride + kh * kKHalf +
                                               ((lane >> 3) & 1) * 8]);
#pragma unroll 6
      for (int ks = 0; ks < kKHalf / 16; ++ks) {
        uint32_t af[4], bf[2];
        ldsm_x4(qa + ks * 32, af);
        ldsm_x2(kb + ks * 32, bf);
        mma_bf16(c, af, bf[0], bf[1]);
      }
      float* sp = sm.sp[kh];
      const int row = hh * 16 + g, col = nt * 8 + 2 * t4;
      sp[row * kSpStride + col] = c[0];
      sp[row * kSpStride + col + 1] = c[1];
      sp[(row + 8) * kSpStride + col] = c[2];
      sp[(row + 8) * kSpStride + col + 1] = c[3];
    }
    __syncthreads();

    // ---- online softmax (exp2 domain) and O += P V --------------------------
    {
      const int R0 = hh2 * 16 + g, R1 = R0 + 8;
      const int cols[4] = {2 * t4, 2 * t4 + 1, 2 * t4 + 8, 2 * t4 + 9};
      float x0[4], x1[4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int cc = cols[u];
        const bool v = sm.tokv[buf][cc] != 0;
        x0[u] = v ? (sm.sp[0][R0 * kSpStride + cc] + sm.sp[1][R0 * kSpStride + cc]) * a.c2
                  : -INFINITY;
        x1[u] = v ? (sm.sp[0][R1 * kSpStride + cc] + sm.sp[1][R1 * kSpStride + cc]) * a.c2
                  : -INFINITY;
        mx0 = fmaxf(mx0, x0[u]);
        mx1 = fmaxf(mx1, x1[u]);
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
      float e0[4], e1[4], p0[4], p1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        e0[u] = exp2f(x0[u] - ref0);
        e1[u] = exp2f(x1[u] - ref1);
      }
      uint32_t pa[4];
      pa[0] = pack_bf16(e0[0], e0[1]);
      pa[1] = pack_bf16(e1[0], e1[1]);
      pa[2] = pack_bf16(e0[2], e0[3]);
      pa[3] = pack_bf16(e1[2], e1[3]);
      {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(pa);
        const float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
        const float2 f2 = __bfloat1622float2(h[2]), f3 = __bfloat1622float2(h[3]);
        p0[0] = f0.x; p0[1] = f0.y; p0[2] = f2.x; p0[3] = f2.y;
        p1[0] = f1.x; p1[1] = f1.y; p1[2] = f3.x; p1[3] = f3.y;
      }
      float s0 = e0[0] + e0[1] + e0[2] + e0[3], s1 = e1[0] + e1[1] + e1[2] + e1[3];
      float r0 = p0[0] + p0[1] + p0[2] + p0[3], r1 = p1[0] + p1[1] + p1[2] + p1[3];
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
#pragma unroll
      for (int j = 0; j < kDv / 4 / 8; ++j) {
        acc[j][0] *= al0;
        acc[j][1] *= al0;
        acc[j][2] *= al1;
        acc[j][3] *= al1;
      }
      const uint32_t vb = smem_u32(&sm.kv[buf][((lane & 7) + ((lane >> 3) & 1) * 8) * kStride +
                                               dq * (kDv / 4) + (lane >> 4) * 8]);
#pragma unroll
      for (int jj = 0; jj < kDv / 4 / 16; ++jj) {
        uint32_t bf[4];
        ldsm_x4_t(vb + jj * 32, bf);
        mma_bf16(acc[2 * jj], pa, bf[0], bf[1]);
        mma_bf16(acc[2 * jj + 1], pa, bf[2], bf[3]);
      }
    }
  }
  if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);

  // ---- O / l in bf16, lse2 = m + log2 l --------------------------------------
  const float inv0 = w0 > 0.f ? 1.f / w0 : 0.f, inv1 = w1 > 0.f ? 1.f / w1 : 0.f;
  __nv_bfloat16* o0 = a.out + (obase + h_lo) * kDv + dq * (kDv / 4) + 2 * t4;
  __nv_bfloat16* o1 = o0 + 8 * kDv;
#pragma unroll
  for (int j = 0; j < kDv / 4 / 8; ++j) {
    *reinterpret_cast<uint32_t*>(o0 + j * 8) = pack_bf16(acc[j][0] * inv0, acc[j][1] * inv0);
    *reinterpret_cast<uint32_t*>(o1 + j * 8) = pack_bf16(acc[j][2] * inv1, acc[j][3] * inv1);
  }
  if (dq == 0 && t4 == 0) {
    a.lse2[obase + h_lo] = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
    a.lse2[obase + h_lo + 8] = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
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
