// The step kernels with the candidate buffer in library-owned device memory.
//
// dsa_indexer_steps_noalloc runs dsa_shard_topk_pack, dsa_merge_topk_stable
// and dsa_convert_index_compact, unchanged, with the packed candidates
// ([rows][S*K][2] fp32) in a static device array of this library instead of a
// caller buffer, for callers that cannot allocate one.  Every argument of the
// three calls is checked before the first kernel is queued.  The array's
// address is looked up on every call (a host-side table lookup), so it stays
// right when the module is loaded again in a new context.  Calls that share a
// device share the array, so they must not overlap in time (one stream, or
// ordered streams).
#include "checks.h"
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_cand_scratch[kScratchBytes];

// Address of the array in the current context (nullptr if the lookup fails).
float* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_cand_scratch) != cudaSuccess) return nullptr;
  return static_cast<float*>(p);
}

}  // namespace

extern "C" dsa_status dsa_indexer_steps_noalloc(const float* logits, int64_t ld, int rows,
                                                int S, int I, int K,
                                                const int32_t* row_starts,
                                                const int32_t* row_ends,
                                                const int32_t* block_table, int reqs,
                                                int max_blocks, int block_size,
                                                const int32_t* row_to_req, int32_t* ids,
                                                int32_t* slots, int32_t* counts,
                                                uint32_t* err_flags, cudaStream_t stream) {
  // The array's size limit and every check of the three calls first, so that
  // a bad argument queues nothing.  The array stands in for the candidate
  // pointer: it is 256-byte aligned, so any non-null, 16-byte-aligned value
  // checks the same way.
  if (rows > 0 && S > 0 && K > 0 &&
      (uint64_t)rows * (uint64_t)S * (uint64_t)K * 8u > kScratchBytes)
    return DSA_ERR_UNSUPPORTED;
  const float* cand_probe = reinterpret_cast<const float*>(uintptr_t{256});
  dsa_status st = dsa::check_shard_topk_pack(logits, ld, rows, S, I, K, row_ends, cand_probe);
  if (st != DSA_OK) return st;
  st = dsa::check_merge_topk_stable(cand_probe, rows, S * K, K, ids);
  if (st != DSA_OK) return st;
  st = dsa::check_convert_index_compact(ids, rows, K, S, I, block_table, reqs, max_blocks,
                                        block_size, slots);
  if (st != DSA_OK) return st;
  if (rows == 0) return DSA_OK;
  float* cand = scratch_on_current_device();
  if (!cand) return DSA_ERR_CUDA;
  st = dsa_shard_topk_pack(logits, ld, rows, S, I, K, row_starts, row_ends, nullptr, cand,
                           err_flags, stream);
  if (st != DSA_OK) return st;
  st = dsa_merge_topk_stable(cand, rows, S * K, K, ids, nullptr, err_flags, stream);
  if (st != DSA_OK) return st;
  return dsa_convert_index_compact(ids, rows, K, S, I, block_table, reqs, max_blocks, block_size,
                                   row_to_req, slots, counts, err_flags, stream);
}
