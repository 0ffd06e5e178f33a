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
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvWarps = kConvThreads / 32;
constexpr int kMaxChunks = 2048 / kConvThreads;   // 32-id chunks per warp for K <= 2048

__global__ void __launch_bounds__(kConvThreads)
    convert_kernel(const int32_t* __restrict__ ids, int rows, int K, int S, int I,
                   const int32_t* __restrict__ bt, int reqs, int max_blocks, int bs,
                   const int32_t* __restrict__ row_to_req, int32_t* __restrict__ slots,
                   int32_t* __restrict__ counts, uint32_t* flags) {
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

  int id_c[kMaxChunks], own_c[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < nch) {
      const int id = mine[c * 32 + lane];
      const int o = id >= 0 ? (int)owner_of(id, S, I) : -1;
      id_c[c] = id;
      own_c[c] = o;
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
  __syncthreads();

  // Issue every block-table load of this warp before the dependent compaction.
  bool bad = !req_ok;
  int slot_c[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    slot_c[c] = -1;
    if (c < nch && own_c[c] >= 0) {
      const int id = id_c[c], o = own_c[c];
      const int64_t l = local_slot_of(id, S, I);
      const int64_t col = l / bs;
      if (req_ok && col < max_blocks) {
        const int blk = __ldg(bt + ((int64_t)o * reqs + req) * max_blocks + col);
        const int64_t v = (int64_t)blk * bs + l % bs;
        if (blk >= 0 && v <= (int64_t)INT32_MAX) slot_c[c] = (int)v;
        else bad = true;
      } else {
        bad = true;
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    if (c < nch) {
      const int o = own_c[c], slot = slot_c[c];
      const unsigned peers = __match_any_sync(kFull, o);
      if (o >= 0) slots[((int64_t)o * rows + r) * K + cnt[warp][o] + __popc(peers & lt)] = slot;
      __syncwarp();
      if (o >= 0 && lane == __ffs(peers) - 1) cnt[warp][o] += __popc(peers);
      __syncwarp();
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);

  // -1 after each shard's valid slots.
  for (int s = 0; s < S; ++s) {
    int32_t* dst = slots + ((int64_t)s * rows + r) * K;
    for (int j = total[s] + tid; j < K; j += kConvThreads) dst[j] = -1;
  }
  if (counts)
    for (int s = tid; s < S; s += kConvThreads) counts[(int64_t)s * rows + r] = total[s];
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_convert_index_compact(const int32_t* ids, int rows, int K, int S,
                                                int I, const int32_t* block_table, int reqs,
                                                int max_blocks, int block_size,
                                                const int32_t* row_to_req, int32_t* slots,
                                                int32_t* counts, uint32_t* err_flags,
                                                cudaStream_t stream) {
  if (rows < 0 || reqs < 1 || max_blocks < 1 || block_size < 1) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!ids || !block_table || !slots) return DSA_ERR_INVALID_ARG;
  convert_kernel<<<rows, kConvThreads, 0, stream>>>(ids, rows, K, S, I, block_table, reqs,
                                                    max_blocks, block_size, row_to_req, slots,
                                                    counts, err_flags);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
