// The step kernels with the candidate buffer in library-owned device memory.
//
// dsa_indexer_steps_noalloc runs dsa_shard_topk_pack, dsa_merge_topk_stable
// and dsa_convert_index_compact, unchanged, with the packed candidates
// ([rows][S*K][2] fp32) in a static device array of this library instead of a
// caller buffer, for callers that cannot allocate one.  The array's address is
// looked up once per device.  Calls that share a device share the array, so
// they must not overlap in time (one stream, or ordered streams).
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_cand_scratch[kScratchBytes];

// Address of the array on the current device, looked up on first use.
float* scratch_on_current_device() {
  constexpr int kMaxDevices = 64;
  static float* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cand_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<float*>(p);
  }
  return ptrs[dev];
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
  if (rows < 0 || S < 1 || K < 1) return rows < 0 ? DSA_ERR_INVALID_ARG : DSA_ERR_UNSUPPORTED;
  if ((uint64_t)rows * (uint64_t)S * (uint64_t)K * 8u > kScratchBytes) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  float* cand = scratch_on_current_device();
  if (!cand) return DSA_ERR_CUDA;
  dsa_status st = dsa_shard_topk_pack(logits, ld, rows, S, I, K, row_starts, row_ends, nullptr,
                                      cand, err_flags, stream);
  if (st != DSA_OK) return st;
  st = dsa_merge_topk_stable(cand, rows, S * K, K, ids, nullptr, err_flags, stream);
  if (st != DSA_OK) return st;
  return dsa_convert_index_compact(ids, rows, K, S, I, block_table, reqs, max_blocks, block_size,
                                   row_to_req, slots, counts, err_flags, stream);
}
