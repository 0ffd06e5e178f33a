// Write-side slot mapping of new tokens under DCP.
//
// PR #40996 report, "DCP supports hybrid attention", section 实现拆解 item 2
// (a per-rank token -> KV-slot mapping over rank-local block tables whose
// allocation blocks hold KV_CACHE_BLOCK_SIZE tokens) and item 1 (a rank keeps
// only its share of each sequence); the ownership rule of the PR #46076
// report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE", section
// 关键源码片段 (`_dcp_localize_decode_seq_lens`).
//
// Token i at global position t of request q is stored by shard owner(t) at
// its local slot l, through that shard's own table row:
// tables[owner][q][l / bs] * bs + l mod bs.  Every other shard's entry for
// the token is -1 (a cache insert skips it).  This is the inverse of the
// read-side conversion in convert.cu: a merged id maps to the slot its token
// was written to.  One thread per token; each shard's output row is written
// with coalesced stores.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kSmThreads = 256;

__global__ void __launch_bounds__(kSmThreads)
    slot_mapping_kernel(const int32_t* __restrict__ positions,
                        const int32_t* __restrict__ token_req, int n, int S,
                        const int32_t* __restrict__ bt, int reqs, int max_blocks, int bs,
                        int32_t* __restrict__ out, uint32_t* flags, const ShardMath sh,
                        const FastDiv fbs) {
  const int i = blockIdx.x * kSmThreads + threadIdx.x;
  if (i >= n) return;
  const int t = __ldg(positions + i);
  int owner = -1;
  int32_t slot = -1;
  bool bad = false;
  if (t >= 0) {   // a negative position is a padding token
    owner = sh.owner((uint32_t)t);
    uint32_t off;
    const uint32_t col = fdivmod(sh.local_slot((uint32_t)t), fbs, &off);
    const int req = token_req ? __ldg(token_req + i) : i;
    if (req >= 0 && req < reqs && col < (uint32_t)max_blocks) {
      const int32_t b = __ldg(bt + ((int64_t)owner * reqs + req) * max_blocks + col);
      const int64_t v = (int64_t)b * bs + off;
      if (b >= 0 && v <= (int64_t)INT32_MAX) slot = (int32_t)v;
      else bad = true;
    } else {
      bad = true;
    }
  }
  for (int s = 0; s < S; ++s) out[(int64_t)s * n + i] = s == owner ? slot : -1;
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_slot_mapping(const int32_t* positions, const int32_t* token_req, int n,
                                       int S, int I, const int32_t* block_table, int reqs,
                                       int max_blocks, int block_size, int32_t* slot_mapping,
                                       uint32_t* err_flags, cudaStream_t stream) {
  if (n < 0 || reqs < 1 || max_blocks < 1 || block_size < 1) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)I * S > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (n == 0) return DSA_OK;
  if (!positions || !block_table || !slot_mapping) return DSA_ERR_INVALID_ARG;
  const unsigned blocks = (unsigned)((n + kSmThreads - 1) / kSmThreads);
  const cudaError_t e = launch_kernel(slot_mapping_kernel, dim3(blocks), dim3(kSmThreads), 0,
                                      stream, 0, positions, token_req, n, S, block_table, reqs,
                                      max_blocks, block_size, slot_mapping, err_flags,
                                      ShardMath(S, I), FastDiv((uint32_t)block_size));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
