// Indexer logits on the fifth-generation tensor cores (sm_103a): for each
// shard s and query row r, every local slot l of r's range on s gets
//
//   logit = sum_h w[r][h] * max(0, q[r][h] . k_s[slot(l)]),
//
// with 64 fp8 (e4m3) query heads of 128 values, fp32 head weights and shard
// s's paged fp8 key cache (PR #46076 report, "[Attention][DSA] support dcp for
// FLASHINFER_MLA_SPARSE", section 关键源码片段: the fp32 indexer logits that
// reach the DCP top-K, each rank scoring its local KV shard; the head sum is
// the DeepSeek-V3.2-style indexer reading of that step).
//
// One CTA per (shard, row, chunk of 16 tiles of 128 local slots), six warps:
//   warp 4   TMA producer: the row's 64 query heads once (8 KB), then per tile
//            the 128 keys, one 2-D tensor copy per block of the paged cache
//            (a 64-row box for 64-token blocks), into a 4-stage ring; the
//            copies use the 128-byte swizzle that the MMA descriptors name.
//            Warp 4 also allocates and frees the tensor memory.
//   warp 5   MMA issuer (one thread): per tile, D[128 tokens][64 heads] =
//            K_tile . Q^T as four tcgen05.mma kind::f8f6f4 (K = 32 each) into
//            one of two 64-column fp32 accumulators in tensor memory; a commit
//            frees the key stage, another hands the accumulator to the
//            epilogue.
//   warps 0-3  epilogue: warp w reads tensor-memory lanes 32w..32w+31 (one
//            token per thread, 64 head sums), applies ReLU and the head
//            weights, and stores the logit (a warp writes 32 consecutive
//            slots); then it releases the accumulator.
// Every wait is bounded: a wait that runs out raises DSA_FLAG_TIMEOUT, the
// roles stop, drain their copies and MMAs (bounded) and the tensor memory is
// freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kHeads = DSA_IDX_HEADS;      // 64
constexpr int kDim = DSA_IDX_DIM;          // 128 fp8 values = 128 bytes per row
constexpr int kTile = 128;                 // tokens per tile = MMA M
constexpr int kStages = 4;
constexpr int kTilesPerCta = 16;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 128;        // two 64-column accumulators
constexpr uint32_t kTileBytes = kTile * kDim;
constexpr uint32_t kQBytes = kHeads * kDim;

struct alignas(1024) LogitsSmem {
  uint8_t k[kStages][kTileBytes];          // 1024-aligned: the swizzle atom
  uint8_t q[kQBytes];
  float w[kHeads];
  uint64_t full[kStages], empty[kStages], qfull, accfull[2], accempty[2], drain;
  uint32_t tmem;
  int abort;
};

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A and B e4m3 (format 0), both K-major, N = 64 (bits 17-22: N >> 3),
// M = 128 (bits 24-28: M >> 4).
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kHeads >> 3) << 17) |
                            ((uint32_t)(kTile >> 4) << 24);

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: start
// address >> 4 (bits 0-13), leading offset (unused here, 1), stride between
// 8-row groups 1024 bytes >> 4 (bits 32-45), descriptor version 1 (bits
// 46-47), swizzle mode 2 = 128 bytes (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
  const uint32_t a = smem_u32(p);
  return (uint64_t)((a >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accum)
      : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 64 consecutive fp32 columns of this warp's 32 tensor-memory lanes (four
// 16-column loads, then one wait).  The wait names every destination register
// as read and written, so no use of them can be scheduled before it.
#define DSA_TMEM_LD16(o)                                                                    \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, "  \
               "%8, %9, %10, %11, %12, %13, %14, %15}, [%16];"                              \
               : "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]),           \
                 "=r"(r[o + 4]), "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7]),           \
                 "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]), "=r"(r[o + 11]),         \
                 "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15])        \
               : "r"(taddr + (uint32_t)(o)))
#define DSA_WAIT_LD16(o)                                                                    \
  asm volatile(""                                                                           \
               : "+r"(r[o + 0]), "+r"(r[o + 1]), "+r"(r[o + 2]), "+r"(r[o + 3]),           \
                 "+r"(r[o + 4]), "+r"(r[o + 5]), "+r"(r[o + 6]), "+r"(r[o + 7]),           \
                 "+r"(r[o + 8]), "+r"(r[o + 9]), "+r"(r[o + 10]), "+r"(r[o + 11]),         \
                 "+r"(r[o + 12]), "+r"(r[o + 13]), "+r"(r[o + 14]), "+r"(r[o + 15]))

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  DSA_TMEM_LD16(0);
  DSA_TMEM_LD16(16);
  DSA_TMEM_LD16(32);
  DSA_TMEM_LD16(48);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  // Empty statements that read and write every destination after the wait.
  DSA_WAIT_LD16(0);
  DSA_WAIT_LD16(16);
  DSA_WAIT_LD16(32);
  DSA_WAIT_LD16(48);
}
#undef DSA_TMEM_LD16
#undef DSA_WAIT_LD16

__device__ __forceinline__ bool aborted(const LogitsSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

__global__ void __launch_bounds__(kThreads, 2)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_q, const float* __restrict__ w,
                          const int32_t* __restrict__ block_table, int reqs, int max_blocks,
                          int block_size, int box_rows, int64_t n_slots,
                          const int32_t* __restrict__ row_to_req,
                          const int32_t* __restrict__ row_starts,
                          const int32_t* __restrict__ row_ends, int rows, int S, int64_t ld,
                          int chunks, float* __restrict__ logits, uint32_t* flags,
                          const ShardMath sh) {
  extern __shared__ unsigned char logits_smem_raw[];
  LogitsSmem& sm = *reinterpret_cast<LogitsSmem*>(
      (reinterpret_cast<uintptr_t>(logits_smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x % chunks;
  const int sr = blockIdx.x / chunks;
  const int s = sr / rows, r = sr - s * rows;

  // This row's local range on shard s (clipped to ld, as the local top-K does).
  int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  int64_t lo = sh.local_len((uint32_t)st, s), hi = sh.local_len((uint32_t)en, s);
  if (hi > ld) { hi = ld; bad = true; }
  if (lo > hi) { lo = hi; bad = true; }
  if (bad && tid == 0 && c == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
  const int64_t t_lo = max(lo / kTile, (int64_t)c * kTilesPerCta);
  const int64_t t_hi = min((hi + kTile - 1) / kTile, (int64_t)(c + 1) * kTilesPerCta);
  const int ntiles = (int)max((int64_t)0, t_hi - t_lo);
  if (ntiles == 0) return;   // same in every thread

  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32 * 5) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(&sm.qfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.accfull[b], 1);
      mbar_init(&sm.accempty[b], 4);   // one arrival per epilogue warp
    }
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    mbar_init_fence();
  }
  if (tid < kHeads) sm.w[tid] = w[(int64_t)r * kHeads + tid];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const int req = row_to_req ? row_to_req[r] : r;

  if (warp == 4) {
    // ---- producer ---------------------------------------------------------
    if (lane == 0) {
      mbar_expect_tx(&sm.qfull, kQBytes);
      tma_load_2d(sm.q, &tm_q, 0, r * kHeads, &sm.qfull);
      const bool req_ok = req >= 0 && req < reqs;
      if (!req_ok) raise_flag(flags, DSA_FLAG_BOUNDS);
      const int32_t* bt = block_table + ((int64_t)s * reqs + (req_ok ? req : 0)) * max_blocks;
      const int oob_y = (int)((int64_t)S * n_slots);   // past the cache: zero fill
      int issued = 0;
      for (int k = 0; k < ntiles; ++k) {
        const int stg = k % kStages;
        if (k >= kStages && !mbar_wait(&sm.empty[stg], (uint32_t)((k / kStages) - 1) & 1u)) {
          raise_flag(flags, DSA_FLAG_TIMEOUT);
          sm.abort = 1;
          break;
        }
        if (aborted(sm)) break;
        mbar_expect_tx(&sm.full[stg], kTileBytes);
        const int64_t tok0 = (t_lo + k) * kTile;
        for (int j = 0; j < kTile / box_rows; ++j) {
          const int64_t l0 = tok0 + (int64_t)j * box_rows;   // first local slot of the box
          const int64_t blk = l0 / block_size, off = l0 - blk * block_size;
          int y = oob_y;
          if (req_ok && l0 < hi && blk < max_blocks) {
            const int64_t p = bt[blk];
            if (p >= 0 && p * block_size + off + box_rows <= n_slots)
              y = (int)((int64_t)s * n_slots + p * block_size + off);
            else
              raise_flag(flags, DSA_FLAG_BOUNDS);
          }
          tma_load_2d(sm.k[stg] + (uint32_t)j * box_rows * kDim, &tm_k, 0, y, &sm.full[stg]);
        }
        ++issued;
      }
      // Drain: every issued tile's copies have landed before the CTA can exit.
      mbar_wait(&sm.qfull, 0);
      for (int k = max(0, issued - kStages); k < issued; ++k)
        mbar_wait(&sm.full[k % kStages], (uint32_t)(k / kStages) & 1u);
    }
  } else if (warp == 5) {
    // ---- MMA issuer -------------------------------------------------------
    if (lane == 0) {
      bool ok = mbar_wait(&sm.qfull, 0);
      const uint64_t qdesc = sw128_desc(sm.q);
      for (int k = 0; ok && k < ntiles; ++k) {
        const int stg = k % kStages, b = k & 1;
        if (k >= 2 && !mbar_wait(&sm.accempty[b], (uint32_t)((k >> 1) - 1) & 1u)) { ok = false; break; }
        if (!mbar_wait(&sm.full[stg], (uint32_t)(k / kStages) & 1u)) { ok = false; break; }
        if (aborted(sm)) break;
        tc_fence_after();
        const uint64_t kdesc = sw128_desc(sm.k[stg]);
#pragma unroll
        for (int kk = 0; kk < kDim / 32; ++kk)   // 32 fp8 = 32 bytes = 2 descriptor units
          mma_f8(tmem + (uint32_t)b * kHeads, kdesc + 2u * kk, qdesc + 2u * kk, kk > 0);
        mma_commit(&sm.empty[stg]);
        mma_commit(&sm.accfull[b]);
      }
      if (!ok) {
        raise_flag(flags, DSA_FLAG_TIMEOUT);
        sm.abort = 1;
      }
      // Drain: every MMA issued has completed before the tensor memory is freed.
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0);
    }
  } else {
    // ---- epilogue: warps 0-3, one token per thread --------------------------
    float wr[kHeads];
#pragma unroll
    for (int h = 0; h < kHeads; ++h) wr[h] = sm.w[h];
    float* out = logits + ((int64_t)s * rows + r) * ld;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int k = 0; k < ntiles; ++k) {
      const int b = k & 1;
      if (!mbar_wait(&sm.accfull[b], (uint32_t)(k >> 1) & 1u)) {
        if (lane == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
        sm.abort = 1;
        break;
      }
      if (aborted(sm)) break;
      tc_fence_after();
      uint32_t v[kHeads];
      tmem_ld64(tmem + lane_base + (uint32_t)(b * kHeads), v);
      float acc = 0.f;
#pragma unroll
      for (int h = 0; h < kHeads; ++h) acc = fmaf(wr[h], fmaxf(__uint_as_float(v[h]), 0.f), acc);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&sm.accempty[b]);
      const int64_t l = (t_lo + k) * kTile + warp * 32 + lane;
      if (l >= lo && l < hi) out[l] = acc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A 2-D map over rows of 128 bytes, a box of box_rows rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, uint64_t nrows, uint32_t box_rows) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)nrows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDim};
  const cuuint32_t box[2] = {(cuuint32_t)kDim, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_indexer_logits(const uint8_t* q, const float* weights,
                                         const uint8_t* k_cache, int64_t n_slots,
                                         const int32_t* block_table, int reqs, int max_blocks,
                                         int block_size, const int32_t* row_to_req,
                                         const int32_t* row_starts, const int32_t* row_ends,
                                         int rows, int S, int I, float* logits, int64_t ld,
                                         uint32_t* err_flags, cudaStream_t stream) {
  if (rows < 0 || ld < 4 || (ld & 3) || n_slots < 1 || reqs < 1 || max_blocks < 1 ||
      block_size < 1)
    return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  // The key boxes must stay inside one block: 16- or 32-token blocks, or
  // multiples of 64 tokens.
  if (!(block_size == 16 || block_size == 32 || block_size % 64 == 0)) return DSA_ERR_UNSUPPORTED;
  if (ld > (int64_t)INT32_MAX || (int64_t)S * n_slots + 64 > (int64_t)INT32_MAX ||
      (int64_t)rows * kHeads > (int64_t)INT32_MAX || (int64_t)I * S > (int64_t)INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!q || !weights || !k_cache || !block_table || !row_ends || !logits) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || (reinterpret_cast<uintptr_t>(logits) & 3u))
    return DSA_ERR_INVALID_ARG;
  const int box_rows = block_size < 64 ? block_size : 64;
  CUtensorMap tm_k, tm_q;
  if (!encode_rows(&tm_k, k_cache, (uint64_t)S * (uint64_t)n_slots, (uint32_t)box_rows) ||
      !encode_rows(&tm_q, q, (uint64_t)rows * kHeads, (uint32_t)kHeads))
    return DSA_ERR_CUDA;
  const int chunks = (int)((ld + (int64_t)kTile * kTilesPerCta - 1) / ((int64_t)kTile * kTilesPerCta));
  const int64_t blocks = (int64_t)S * rows * chunks;
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  const size_t smem = sizeof(LogitsSmem) + 1024;
  if (cudaFuncSetAttribute(indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const cudaError_t e = launch_kernel(indexer_logits_kernel, dim3((unsigned)blocks),
                                      dim3(kThreads), smem, stream, 0, tm_k, tm_q, weights,
                                      block_table, reqs, max_blocks, block_size, box_rows,
                                      n_slots, row_to_req, row_starts, row_ends, rows, S, ld,
                                      chunks, logits, err_flags, ShardMath(S, I));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
