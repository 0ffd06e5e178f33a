// Merged global ids -> each shard's physical paged-KV slots, compacted.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 实现拆解 item 4 (`_convert_req_index_to_global_index_kernel` with
// DCP_SIZE / DCP_RANK / DCP_INTERLEAVE de-interleaving, and the
// COMPACT_TO_FRONT branch that packs valid slots at the front) and section
// 评论区精华 (the compaction fused into the convert kernel).  PR #40996 report,
// "DCP supports hybrid attention", section 关键源码片段: block tables are
// rank-local, so shard s maps its own local position through its own table.
//
// The pages place valid slots with an atomic counter, which leaves their order
// open.  Here every shard's slots keep the merged (rank) order: one CTA per
// row, each warp owns a contiguous piece of the id list, counts per shard,
// the CTA takes an exclusive scan over warps, and each warp then writes its
// ids at their final positions using match_any peer groups.
#include "checks.h"
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvWarps = kConvThreads / 32;
constexpr int kMaxChunks = 2048 / kConvThreads;   // 32-id chunks per warp for K <= 2048

__global__ void __launch_bounds__(kConvThreads)
    convert_kernel(const int32_t* __restrict__ ids, int rows, int K, int S,
                   const int32_t* __restrict__ bt, int reqs, int max_blocks, int bs,
                   const int32_t* __restrict__ row_to_req, int32_t* __restrict__ slots,
                   int32_t* __restrict__ counts, uint32_t* flags, const ShardMath sh,
                   const FastDiv fbs) {
  __shared__ int cnt[kConvWarps][DSA_MAX_SHARDS];
  __shared__ int total[DSA_MAX_SHARDS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  for (int i = tid; i < kConvWarps * DSA_MAX_SHARDS; i += kConvThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();

  const int req = row_to_req ? row_to_req[r] : r;
  const bool req_ok = req >= 0 && req < reqs;
  const int seg = K / kConvWarps;          // multiple of 32
  const int nch = seg / 32;
  const int32_t* mine = ids + (int64_t)r * K + warp * seg;
  const unsigned lt = lanemask_lt();

  // Pass 1: owner and local slot of every id; per-warp counts per shard.
  int own_c[kMaxChunks];
  uint32_t loc_c[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    own_c[c] = -1;
    loc_c[c] = 0;
    if (c < nch) {
      const int id = __ldg(mine + c * 32 + lane);
      if (id >= 0) {
        own_c[c] = sh.owner((uint32_t)id);
        loc_c[c] = sh.local_slot((uint32_t)id);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < nch) {
      const int o = own_c[c];
      const unsigned peers = __match_any_sync(kFull, o);
      if (o >= 0 && lane == __ffs(peers) - 1) cnt[warp][o] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int s = tid; s < S; s += kConvThreads) {
    int run = 0;
    for (int w = 0; w < kConvWarps; ++w) {
      const int c = cnt[w][s];
      cnt[w][s] = run;
      run += c;
    }
    total[s] = run;
  }

  // Every block-table load of this thread is issued before the compaction.
  bool bad = !req_ok;
  int slot_c[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    slot_c[c] = -1;
    if (c < nch && own_c[c] >= 0) {
      uint32_t off;
      const uint32_t col = fdivmod(loc_c[c], fbs, &off);
      if (req_ok && col < (uint32_t)max_blocks) {
        const int blk = __ldg(bt + ((int64_t)own_c[c] * reqs + req) * max_blocks + col);
        const int64_t v = (int64_t)blk * bs + off;
        if (blk >= 0 && v <= (int64_t)INT32_MAX) slot_c[c] = (int)v;
        else bad = true;
      } else {
        bad = true;
      }
    }
  }
  __syncthreads();
  // Pass 2: each id at its final position (merged order within its shard).
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < nch) {
      const int o = own_c[c];
      const unsigned peers = __match_any_sync(kFull, o);
      if (o >= 0) slots[((int64_t)o * rows + r) * K + cnt[warp][o] + __popc(peers & lt)] = slot_c[c];
      __syncwarp();
      if (o >= 0 && lane == __ffs(peers) - 1) cnt[warp][o] += __popc(peers);
      __syncwarp();
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);

  // -1 after each shard's valid slots, 16 bytes per store where aligned.
  for (int s = 0; s < S; ++s) {
    int32_t* dst = slots + ((int64_t)s * rows + r) * K;
    const int t0 = total[s];
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      const int a0 = min(K, (t0 + 3) & ~3);
      if (tid < a0 - t0) dst[t0 + tid] = -1;
      int4* d4 = reinterpret_cast<int4*>(dst + a0);
      for (int j = tid; j < (K - a0) / 4; j += kConvThreads) d4[j] = make_int4(-1, -1, -1, -1);
    } else {
      for (int j = t0 + tid; j < K; j += kConvThreads) dst[j] = -1;
    }
  }
  if (counts)
    for (int s = tid; s < S; s += kConvThreads) counts[(int64_t)s * rows + r] = total[s];
}

// ---------------------------------------------------------------------------
// Few shards (S <= 8): one CTA per row (128 threads, or 512 for a batch that
// fits one wave), each warp owning a contiguous piece of the id list in
// chunks of 32.  One pass computes every id's owner and physical slot and,
// per chunk, its position among the warp's ids of the same shard: a ballot per
// shard, the lane's own shard's ballot counted below it, plus that shard's
// running count (held by lane s and read with a shuffle).  A scan over the
// warps' per-shard totals then gives final positions.
// ---------------------------------------------------------------------------
constexpr int kCvMaxS = 8;
constexpr int kCvMaxK = 2048;

// id -> (owner, local slot / block size, local slot mod block size).  When S,
// I and the block size are powers of two (kPow2) the divisions are shifts by
// the log2 sizes held in the divisors' shift fields.
template <bool kPow2>
__device__ __forceinline__ void map_id(uint32_t id, const ShardMath& sh, const FastDiv& fbs,
                                       int* owner, uint32_t* col, uint32_t* off) {
  if (kPow2) {
    const uint32_t lI = sh.fI.l, lS = sh.fS.l, lb = fbs.l;
    *owner = (int)((id >> lI) & (uint32_t)(sh.S - 1));
    const uint32_t local = ((id >> (lI + lS)) << lI) | (id & (uint32_t)(sh.I - 1));
    *col = local >> lb;
    *off = local & (fbs.d - 1u);
  } else {
    *owner = sh.owner(id);
    *col = fdivmod(sh.local_slot(id), fbs, off);
  }
}

// NT threads per row: 128 for large batches, 512 for batches that fit one wave
// (where a row's latency sets the time).
template <int NT, bool kPow2>
__global__ void __launch_bounds__(NT)
    convert_few_kernel(const int32_t* __restrict__ ids, int rows, int K, int S,
                       const int32_t* __restrict__ bt, int reqs, int max_blocks, int bs,
                       const int32_t* __restrict__ row_to_req, int32_t* __restrict__ slots,
                       int32_t* __restrict__ counts, uint32_t* flags, const ShardMath sh,
                       const FastDiv fbs) {
  constexpr int kCvWarps = NT / 32;
  constexpr int kCvMaxChunks = kCvMaxK / NT;   // chunks of 32 ids per warp for K = 2048
  __shared__ int wbase[kCvWarps][kCvMaxS];   // per-warp counts, then exclusive bases
  __shared__ int total[kCvMaxS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x;
  const int req = row_to_req ? __ldg(row_to_req + r) : r;
  const bool req_ok = req >= 0 && req < reqs;
  const int nch = K / NT;                    // chunks per warp
  const int32_t* mine = ids + (int64_t)r * K + warp * nch * 32;
  const unsigned lt = lanemask_lt();

  // aux_c: the id, then the id's offset inside its block.
  int aux_c[kCvMaxChunks];
#pragma unroll
  for (int c = 0; c < kCvMaxChunks; ++c) aux_c[c] = c < nch ? __ldg(mine + c * 32 + lane) : -1;

  // Owner and block-table entry (-1: none); every table load is issued before use.
  int own_c[kCvMaxChunks], blk_c[kCvMaxChunks];
  bool bad = !req_ok;
#pragma unroll
  for (int c = 0; c < kCvMaxChunks; ++c) {
    own_c[c] = -1;
    blk_c[c] = -1;
    const int id = aux_c[c];
    if (id >= 0) {
      int o;
      uint32_t col, off;
      map_id<kPow2>((uint32_t)id, sh, fbs, &o, &col, &off);
      own_c[c] = o;
      aux_c[c] = (int)off;
      if (req_ok && col < (uint32_t)max_blocks)
        blk_c[c] = __ldg(bt + ((int64_t)o * reqs + req) * max_blocks + col);
    }
  }
  // Positions among the warp's ids of the same shard, in id order: the lanes
  // whose ids share this lane's shard (one match) give its rank in the
  // chunk, and one-hot 8-bit fields summed over the warp give every shard's
  // count in the chunk (at most 32 each; shards 4-7 in a second sum).
  int run = 0;   // lane s < S: this warp's ids of shard s so far
#pragma unroll
  for (int c = 0; c < kCvMaxChunks; ++c) {
    if (c < nch) {
      const int o = own_c[c];
      const unsigned same = __match_any_sync(kFull, o);
      const uint32_t one = o < 0 ? 0u : 1u << (8 * (o & 3));
      uint32_t cnt = __reduce_add_sync(kFull, o < 4 ? one : 0u);
      if (S > 4) {
        const uint32_t hi = __reduce_add_sync(kFull, o >= 4 ? one : 0u);
        if (lane >= 4) cnt = hi;
      }
      const int base = __shfl_sync(kFull, run, o < 0 ? 0 : o);
      own_c[c] = o < 0 ? -1 : (o | ((base + __popc(same & lt)) << 8));
      if (lane < S) run += (int)((cnt >> (8 * (lane & 3))) & 0xffu);
    }
  }
  if (lane < S) wbase[warp][lane] = run;
  __syncthreads();
  if (tid < S) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < kCvWarps; ++w) {
      const int c = wbase[w][tid];
      wbase[w][tid] = acc;
      acc += c;
    }
    total[tid] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kCvMaxChunks; ++c) {
    const int packed = own_c[c];
    if (c < nch && packed >= 0) {
      const int o = packed & 0xff, pos = wbase[warp][o] + (packed >> 8);
      // A missing or negative table entry, or a slot past INT32_MAX, gives
      // -1 and raises the bounds flag.
      int v = -1;
      const int64_t x = (int64_t)blk_c[c] * bs + aux_c[c];
      if (blk_c[c] >= 0 && x <= (int64_t)INT32_MAX) v = (int)x;
      else bad = true;
      slots[((int64_t)o * rows + r) * K + pos] = v;
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);

  // -1 after each shard's valid slots, 16 bytes per store where aligned.
  for (int s = 0; s < S; ++s) {
    int32_t* dst = slots + ((int64_t)s * rows + r) * K;
    const int t0 = total[s];
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      const int a0 = min(K, (t0 + 3) & ~3);
      if (tid < a0 - t0) dst[t0 + tid] = -1;
      int4* d4 = reinterpret_cast<int4*>(dst + a0);
      for (int j = tid; j < (K - a0) / 4; j += NT) d4[j] = make_int4(-1, -1, -1, -1);
    } else {
      for (int j = t0 + tid; j < K; j += NT) dst[j] = -1;
    }
  }
  if (counts && tid < S) counts[(int64_t)tid * rows + r] = total[tid];
}

}  // namespace
}  // namespace dsa

using namespace dsa;

dsa_status dsa::check_convert_index_compact(const int32_t* ids, int rows, int K, int S, int I,
                                            const int32_t* block_table, int reqs, int max_blocks,
                                            int block_size, const int32_t* slots) {
  if (rows < 0 || reqs < 1 || max_blocks < 1 || block_size < 1) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)I * S > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!ids || !block_table || !slots) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

extern "C" dsa_status dsa_convert_index_compact(const int32_t* ids, int rows, int K, int S,
                                                int I, const int32_t* block_table, int reqs,
                                                int max_blocks, int block_size,
                                                const int32_t* row_to_req, int32_t* slots,
                                                int32_t* counts, uint32_t* err_flags,
                                                cudaStream_t stream) {
  const dsa_status st = check_convert_index_compact(ids, rows, K, S, I, block_table, reqs,
                                                    max_blocks, block_size, slots);
  if (st != DSA_OK || rows == 0) return st;
  if (S <= kCvMaxS) {
    auto pow2 = [](int v) { return (v & (v - 1)) == 0; };
    const bool p2 = pow2(S) && pow2(I) && pow2(block_size);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DSA_ERR_CUDA;
    // Batches that fit one wave are latency-bound: more threads per row.
    const bool wide = rows <= 2 * sms;
    auto kern = wide ? (p2 ? convert_few_kernel<512, true> : convert_few_kernel<512, false>)
                     : (p2 ? convert_few_kernel<128, true> : convert_few_kernel<128, false>);
    const cudaError_t e = launch_kernel(kern, dim3((unsigned)rows), dim3(wide ? 512 : 128), 0, stream,
                                        0, ids, rows, K, S, block_table, reqs, max_blocks,
                                        block_size, row_to_req, slots, counts, err_flags,
                                        ShardMath(S, I), FastDiv((uint32_t)block_size));
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  const cudaError_t e = launch_kernel(convert_kernel, dim3((unsigned)rows), dim3(kConvThreads), 0,
                                      stream, 0, ids, rows, K, S, block_table, reqs, max_blocks,
                                      block_size, row_to_req, slots, counts, err_flags,
                                      ShardMath(S, I), FastDiv((uint32_t)block_size));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
