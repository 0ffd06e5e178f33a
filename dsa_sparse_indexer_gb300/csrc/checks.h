// Host-side argument checks of the step entry points, callable on their own.
//
// Each returns what its entry point would return for the same arguments
// before launching anything: DSA_OK when the call would go ahead (or, with
// rows == 0, do nothing), else DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED.
// Scalar arguments are checked first; with rows == 0 pointers are not read.
#pragma once

#include <cstdint>

#include "dsa.h"

namespace dsa {

// dsa_shard_topk_pack (local_idx may be NULL; cand is required).
dsa_status check_shard_topk_pack(const float* logits, int64_t ld, int rows, int S, int I, int K,
                                 const int32_t* row_ends, const float* cand);

// dsa_merge_topk_stable.
dsa_status check_merge_topk_stable(const float* cand, int rows, int C, int K, const int32_t* ids);

// dsa_convert_index_compact.
dsa_status check_convert_index_compact(const int32_t* ids, int rows, int K, int S, int I,
                                       const int32_t* block_table, int reqs, int max_blocks,
                                       int block_size, const int32_t* slots);

}  // namespace dsa
