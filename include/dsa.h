/*
 * dsa.h - C ABI of the DCP sparse-indexer hot path for GB300 (sm_103a).
 *
 * The path, in the order a DCP decode step runs it (PR #46076 report,
 * "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE", section 关键源码片段,
 * `_merge_dcp_topk_global`):
 *
 *   dsa_shard_topk        every shard's local top-K of fp32 indexer logits
 *   dsa_pack_candidates   (score, global id) pairs, written straight into each
 *                         shard's slice of one [rows, S*K, 2] buffer (the
 *                         all_gather of the pages, with no copy)
 *   dsa_merge_topk_stable stable global top-K of the S*K candidates
 *   dsa_convert_index_compact  global ids -> each shard's paged KV slots,
 *                         valid slots compacted to the front
 *   dsa_lse_combine       LSE-weighted combine of the shards' partial
 *                         attention outputs, base-2 LSE converted to base e
 *
 * plus dsa_shard_topk_pack (the first two steps in one kernel),
 * dsa_indexer_fused (the first four steps in one kernel per row, a thread-block
 * cluster of S CTAs exchanging candidates through distributed shared memory)
 * dsa_slot_mapping (the write side of the paged cache: where each shard
 * stores the KV of new tokens) and dsa_sparse_mla_decode (each shard's sparse
 * attention over its compacted slots, whose outputs dsa_lse_combine merges).
 *
 * Sharding (PR #46076 report, section 关键源码片段, comment in
 * `_dcp_localize_decode_seq_lens`): global token t lives on shard
 * owner(t) = (t / I) mod S; a shard keeps its tokens in increasing global
 * order, so t is its local slot loc(t) = (t / (I*S))*I + t mod I, and local
 * slot l of shard s is global token (l / I)*(I*S) + s*I + l mod I.  A global
 * range [start, end) is, on shard s, the local range [n_s(start), n_s(end)),
 * n_s(L) = (L / (I*S))*I + clamp(L mod (I*S) - s*I, 0, I).
 *
 * Ranking everywhere: score descending, ties to the smaller global token id
 * (the "stable" of the pages' selector; -0.0 and +0.0 are the same score).
 * Scores must not be NaN; results for NaN inputs are unspecified.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing, keeps no state between calls and frees nothing (the
 *     one exception, dsa_indexer_steps_noalloc, uses a static device array
 *     that exists while the library is loaded).
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *     enqueues one kernel (dsa_indexer_steps_noalloc: three); results are
 *     ready when the stream reaches it.
 *   - Arguments are checked on the host before anything is enqueued.  A bad
 *     argument returns DSA_ERR_INVALID_ARG or DSA_ERR_UNSUPPORTED and touches
 *     nothing.  rows == 0 returns DSA_OK and enqueues nothing once the scalar
 *     arguments pass (array pointers are then not checked and may be NULL).
 *   - DSA_ERR_CUDA means the launch itself failed (cudaGetLastError).
 *   - Problems only visible on the device set bits of `*err_flags` (a caller
 *     owned device word, may be NULL) with atomicOr; kernels never trap.
 *   - Row-major layouts; int32 indices; -1 marks padding.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment */
  DSA_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels support */
  DSA_ERR_CUDA = 3           /* a CUDA launch error */
} dsa_status;

/* Bits set in *err_flags by the kernels. */
enum {
  DSA_FLAG_BOUNDS = 1u,      /* a row range or block-table column was out of range */
  DSA_FLAG_TIMEOUT = 2u      /* a bounded wait on an async copy ran out */
};

/* Supported top-K sizes: the pages' set, PR #46076 report, section 关键源码片段,
 * `_assert_cutedsl_dcp_merge_supported` (index_topk in 512/1024/2048). */
#define DSA_MAX_SHARDS 64
/* Sparse MLA decode (dsa_sparse_mla_decode): a cache row and a query head are
 * the latent kv_c (DSA_MLA_DV values) followed by the rope part, DSA_MLA_DQK
 * values in all. */
#define DSA_MLA_DQK 576
#define DSA_MLA_DV 512
/* Indexer-logits shape: query heads per token and values per head / key. */
#define DSA_IDX_HEADS 64
#define DSA_IDX_DIM 128

/* Bytes of the library-owned candidate array of dsa_indexer_steps_noalloc. */
#define DSA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Human-readable name of a status code (static string). */
const char* dsa_status_string(dsa_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int dsa_version(void);

/*
 * dsa_shard_topk - every shard's local top-K.
 * PR #46076 report, section 关键源码片段, `_merge_dcp_topk_global` docstring:
 * "topk_indices are top-K positions in this rank's local KV shard".
 *
 *   logits      [S][rows][ld] fp32: shard s, row r, local slot l at
 *               logits[(s*rows + r)*ld + l].  16-byte aligned; ld % 4 == 0.
 *   row_starts  [rows] int32 global start of each row (NULL = all 0)
 *   row_ends    [rows] int32 global end (exclusive) of each row
 *   local_idx   [S][rows][K] int32 out: the K best local slots of
 *               [n_s(start), n_s(end)), ascending; -1 after the first
 *               min(K, n_s(end) - n_s(start)).  Absolute local slots.
 *   err_flags   DSA_FLAG_BOUNDS if a local range ends past ld (the range is
 *               clipped to ld) or starts after it ends (treated as empty);
 *               DSA_FLAG_TIMEOUT if the bounded wait for a row's copy into
 *               shared memory runs out (that (shard, row)'s outputs are then
 *               not written).
 * Errors: S not in [1, 64], I < 1, K not in {512, 1024, 2048} -> UNSUPPORTED;
 *         null pointers, rows < 0, ld < 4, ld % 4, misaligned logits -> INVALID_ARG.
 */
dsa_status dsa_shard_topk(const float* logits, int64_t ld, int rows, int S, int I,
                          int K, const int32_t* row_starts, const int32_t* row_ends,
                          int32_t* local_idx, uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_pack_candidates - (score, global id) candidates of every shard's top-K.
 * PR #46076 report, section 实现拆解 item 1 (`pack_dcp_topk_candidates_cutedsl`)
 * and section 关键源码片段 (packed = [batch, topk, 2] fp32, then all_gather
 * along dim 1).
 *
 *   logits, ld  as dsa_shard_topk
 *   local_idx   [S][rows][K] int32 local slots (-1 = padding), as written by
 *               dsa_shard_topk
 *   cand        [rows][S*K][2] fp32 out.  cand[r][s*K + j] = (logits[s][r][l],
 *               global id of local slot l on shard s) for l = local_idx[s][r][j];
 *               element 1 holds the int32 id's BIT PATTERN (read it back as
 *               int32).  Padding -> (-inf, -1).  16-byte aligned.
 *   err_flags   DSA_FLAG_BOUNDS if a local index is >= ld (written as padding).
 */
dsa_status dsa_pack_candidates(const float* logits, int64_t ld, const int32_t* local_idx,
                               int rows, int S, int I, int K, float* cand,
                               uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_shard_topk_pack - dsa_shard_topk and dsa_pack_candidates in one kernel:
 * the winning logits are packed while still in shared memory, so the pack
 * step's gather from the logits is not repeated.  Same arguments, results and
 * error flags; local_idx may be NULL when only the candidates are wanted.
 */
dsa_status dsa_shard_topk_pack(const float* logits, int64_t ld, int rows, int S, int I,
                               int K, const int32_t* row_starts, const int32_t* row_ends,
                               int32_t* local_idx, float* cand, uint32_t* err_flags,
                               cudaStream_t stream);

/*
 * dsa_merge_topk_stable - the global top-K of each row's C gathered candidates.
 * PR #46076 report, section 实现拆解 item 1
 * (`stable_topk_from_gathered_candidates_cutedsl`) and the
 * `_merge_dcp_topk_global` docstring: topk_indices are overwritten with global
 * token ids, -1 for padding.
 *
 *   cand        [rows][C][2] fp32 candidates as written by the pack; a
 *               candidate whose id is < 0 is padding and never selected.
 *               16-byte aligned; C % 4 == 0; C >= K.
 *   ids         [rows][K] int32 out: the K best valid candidates' ids, best
 *               first; -1 after the valid ones.
 *   scores      [rows][K] fp32 out, may be NULL: their scores (-inf after the
 *               valid ones; a -0.0 score may come back as +0.0).
 *   err_flags   unused (no step of the merge can stall or go out of bounds);
 *               kept so that every step has the same trailing arguments.
 * Candidate ids within a row must be distinct (the pack guarantees it).
 */
dsa_status dsa_merge_topk_stable(const float* cand, int rows, int C, int K,
                                 int32_t* ids, float* scores, uint32_t* err_flags,
                                 cudaStream_t stream);

/*
 * dsa_convert_index_compact - merged global ids -> per-shard physical KV slots.
 * PR #46076 report, section 实现拆解 item 4 (`_convert_req_index_to_global_index_kernel`
 * with DCP_SIZE/DCP_RANK/DCP_INTERLEAVE and the COMPACT_TO_FRONT branch) and
 * PR #40996 report, "DCP supports hybrid attention", section 关键源码片段
 * (rank-local block tables of cdiv(max_len, block_size * cp) columns).
 *
 *   ids         [rows][K] int32 merged ids (-1 = padding)
 *   block_table [S][reqs][max_blocks] int32 physical block numbers per shard
 *   row_to_req  [rows] int32 request of each row (NULL: row r is request r)
 *   slots       [S][rows][K] int32 out: for shard s, the ids it holds, in the
 *               merged order, mapped to block_table[s][req][l / block_size] *
 *               block_size + l % block_size (l = local slot), packed at the
 *               front; -1 after them.  The order is deterministic.
 *   counts      [S][rows] int32 out, may be NULL: number of slots written.
 *   err_flags   DSA_FLAG_BOUNDS if a column is >= max_blocks, a table entry is
 *               negative, a slot does not fit in int32, or a row's request is
 *               outside [0, reqs); such an entry is written as -1 in its place.
 */
dsa_status dsa_convert_index_compact(const int32_t* ids, int rows, int K, int S, int I,
                                     const int32_t* block_table, int reqs, int max_blocks,
                                     int block_size, const int32_t* row_to_req,
                                     int32_t* slots, int32_t* counts, uint32_t* err_flags,
                                     cudaStream_t stream);

/*
 * dsa_indexer_fused - dsa_shard_topk, dsa_pack_candidates, dsa_merge_topk_stable
 * and dsa_convert_index_compact for each row in one kernel, with the same
 * results.  PR #46076 report, section 关键源码片段 (`_merge_dcp_topk_global`:
 * local top-K on every rank, candidate all_gather, stable selector) and section
 * 实现拆解 items 1, 2 and 4.
 *
 * Each row is handled by a thread-block cluster of S CTAs, one per shard; the
 * candidates a shard selects stay in its shared memory and the all_gather of
 * the pages becomes distributed-shared-memory reads inside the cluster, so
 * neither candidates nor merged ids make a round trip through HBM.
 *
 *   logits, ld, rows, S, I, K, row_starts, row_ends   as dsa_shard_topk
 *   block_table, reqs, max_blocks, block_size, row_to_req
 *                    as dsa_convert_index_compact
 *   ids      [rows][K] int32 out, as dsa_merge_topk_stable
 *   scores   [rows][K] fp32 out, may be NULL, as dsa_merge_topk_stable
 *   slots    [S][rows][K] int32 out, counts [S][rows] int32 out (may be NULL),
 *            as dsa_convert_index_compact
 *   local_idx [S][rows][K] int32 out, may be NULL, as dsa_shard_topk
 *   cand     [rows][S*K][2] fp32 out, may be NULL, as dsa_pack_candidates
 *   err_flags as the single-step calls.
 * Errors: as the single-step calls; S > 8 (the portable cluster size) returns
 * DSA_ERR_UNSUPPORTED (use the single-step calls).
 */
dsa_status dsa_indexer_fused(const float* logits, int64_t ld, int rows, int S, int I, int K,
                             const int32_t* row_starts, const int32_t* row_ends,
                             const int32_t* block_table, int reqs, int max_blocks,
                             int block_size, const int32_t* row_to_req, int32_t* ids,
                             float* scores, int32_t* slots, int32_t* counts,
                             int32_t* local_idx, float* cand, uint32_t* err_flags,
                             cudaStream_t stream);

/*
 * dsa_lse_combine - merge the shards' partial attention outputs by their LSE.
 * PR #46076 report, section 实现拆解 item 5 and section 评论区精华 (LSE base
 * normalisation: the sparse MLA kernel's LSE is base 2, the DCP reducer wants
 * base e); PR #52046 report, "DSV3.2 PCP sharding", section 关键源码片段
 * (`dcp_manager.combine(attn_out, lse, ...)`).
 *
 * Per (row, head): lambda_s = lse2_s * ln 2, M = max_s lambda_s,
 * w_s = exp(lambda_s - M), out = sum_s w_s O_s / sum_s w_s, lse = M + ln sum_s w_s.
 * A shard with lse2 = -inf holds nothing and its output is not read; if every
 * shard is -inf the result is out = 0, lse = -inf.
 *
 *   partial_out [S][rows][H][D] bf16 (raw uint16 bit patterns), 16-byte aligned
 *   lse2        [S][rows][H] fp32 base-2 LSE
 *   out         [rows][H][D] bf16 out (round to nearest even), 16-byte aligned
 *   lse_out     [rows][H] fp32 out, base e; may be NULL
 *   err_flags   device word for DSA_FLAG_* bits, may be NULL (no condition of
 *               this kernel currently sets one; kept for a uniform interface).
 * Errors: D % 8 != 0, H < 1, D < 8 -> INVALID_ARG; S not in [1, 64] -> UNSUPPORTED.
 */
dsa_status dsa_lse_combine(const uint16_t* partial_out, const float* lse2, int S,
                           int rows, int H, int D, uint16_t* out, float* lse_out,
                           uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_slot_mapping - where each shard writes the KV of new tokens (the write
 * side of the paged cache; dsa_convert_index_compact is the read side).
 * PR #40996 report, "DCP supports hybrid attention", section 实现拆解 item 2
 * (per-rank token -> KV-slot mapping over rank-local block tables with
 * allocation blocks of KV_CACHE_BLOCK_SIZE tokens) and item 1; the ownership
 * rule of the PR #46076 report, section 关键源码片段.
 *
 * Token i at global position t = positions[i] of request q = token_req[i] is
 * stored by shard s = (t / I) mod S at its local slot l = (t / (I*S))*I +
 * t mod I, i.e. at block_table[s][q][l / block_size] * block_size +
 * l % block_size; every other shard's entry is -1.
 *
 *   positions    [n] int32 global positions; a negative one is a padding token
 *                (-1 on every shard, no error)
 *   token_req    [n] int32 request of each token (NULL: token i is request i)
 *   block_table  [S][reqs][max_blocks] int32 physical block numbers per shard,
 *                in allocation blocks of block_size tokens (a kernel block of
 *                block_size / m tokens inside one does not change the slot)
 *   slot_mapping [S][n] int32 out
 *   err_flags    DSA_FLAG_BOUNDS if a request is outside [0, reqs), a column
 *                is >= max_blocks, a table entry is negative or a slot does not
 *                fit in int32; that token is then -1 on every shard.
 * Errors: n < 0, reqs < 1, max_blocks < 1, block_size < 1, null pointers ->
 *         INVALID_ARG; S not in [1, 64], I < 1, I*S > INT32_MAX -> UNSUPPORTED.
 */
dsa_status dsa_slot_mapping(const int32_t* positions, const int32_t* token_req, int n,
                            int S, int I, const int32_t* block_table, int reqs,
                            int max_blocks, int block_size, int32_t* slot_mapping,
                            uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_sparse_mla_decode - every shard's sparse MLA decode attention over its
 * compacted KV slots: the partial outputs and base-2 LSEs dsa_lse_combine merges.
 * PR #52046 report, "DSV3.2 PCP sharding", section 关键源码片段
 * (`_fused_norm_rope_kernel`: a cache row is the normed latent kv_c followed by
 * the roped k_pe; `_sparse_indexer_and_attn`: the MQA query is its parts
 * concatenated on the last dimension, `forward_mqa(q, kv_cache, ...)` returns
 * output and LSE per shard); PR #46076 report, section 实现拆解 items 4 and 5
 * (compacted slots in, base-2 LSE out).
 *
 * For shard s, row r, head h, over j in slots[s][r][0 .. counts[s][r]):
 *   x_j = scale * (q[r][h] . kv_cache[s][slot_j]),
 *   out[s][r][h] = sum_j exp(x_j) v_j / sum_j exp(x_j),  v_j = first DSA_MLA_DV
 *   entries of the row; lse2[s][r][h] = log2 sum_j exp(x_j).
 * A shard with no slot gives out = 0 and lse2 = -inf.  Scores accumulate in
 * fp32 from bf16 products; the softmax weights enter the value product as bf16.
 *
 *   q          [rows][H][DSA_MLA_DQK] bf16 (uint16 bit patterns), 16-byte aligned
 *   kv_cache   [S][n_slots][DSA_MLA_DQK] bf16, 16-byte aligned: each shard's
 *              paged cache by physical slot (block * block_size + offset)
 *   slots      [S][rows][K] int32, counts [S][rows] int32: the compacted slots
 *              and their number, as dsa_convert_index_compact writes them
 *   scale      softmax scale (finite)
 *   out        [S][rows][H][DSA_MLA_DV] bf16 out, 16-byte aligned
 *   lse2       [S][rows][H] fp32 out
 *   err_flags  DSA_FLAG_BOUNDS if a count is outside [0, K] (clamped) or a slot
 *              below it is outside [0, n_slots) (that token is left out).
 * Errors: rows < 0, K < 1, n_slots < 1, non-finite scale, null pointers,
 *         misalignment -> INVALID_ARG; S not in [1, 64], H not a multiple of
 *         64 -> UNSUPPORTED.
 */
dsa_status dsa_sparse_mla_decode(const uint16_t* q, const uint16_t* kv_cache, int64_t n_slots,
                                 const int32_t* slots, const int32_t* counts, int rows, int S,
                                 int H, int K, float scale, uint16_t* out, float* lse2,
                                 uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_indexer_logits - each shard's indexer logits over its local slots.
 * PR #46076 report, section 关键源码片段: `_assert_cutedsl_dcp_merge_supported`
 * (fp32 indexer logits reach the DCP top-K) and the `_merge_dcp_topk_global`
 * docstring (each rank scores its own local KV shard); PR #52046 report,
 * "DSV3.2 PCP sharding", section 关键源码片段 (`_sparse_indexer_and_attn`: the
 * indexer scores a request's cached keys).  The formula is not printed on the
 * pages; the reading taken is the DeepSeek-V3.2-style indexer:
 *
 *   logits[s][r][l] = sum_h weights[r][h] * max(0, q[r][h] . k_s(l)),
 *
 * k_s(l) the key of shard s's local slot l of row r's request, at physical
 * slot block_table[s][req][l / block_size] * block_size + l % block_size.
 *
 *   q           [rows][DSA_IDX_HEADS][DSA_IDX_DIM] fp8 e4m3 codes, 16-byte aligned
 *   weights     [rows][DSA_IDX_HEADS] fp32
 *   k_cache     [S][n_slots][DSA_IDX_DIM] fp8 e4m3 codes, 16-byte aligned:
 *               each shard's paged key cache by physical slot
 *   block_table [S][reqs][max_blocks] int32; row_to_req [rows] (NULL: row r
 *               is request r); row_starts (NULL = 0) / row_ends [rows] global
 *   logits      [S][rows][ld] fp32 out (4-byte aligned; ld % 4 == 0): entries
 *               l in [n_s(start), n_s(end)) are written, the others untouched
 * Products of fp8 values are exact; each head's 128 of them are summed in
 * fp32 by the tensor cores, then ReLU, weights and the head sum in fp32.
 *   err_flags   DSA_FLAG_BOUNDS if a range ends past ld (clipped), a request
 *               is outside [0, reqs) or a needed table entry points outside the
 *               cache (those keys read as zero); DSA_FLAG_TIMEOUT if a bounded
 *               wait ran out (the CTA stops; its slots are not all written).
 * Errors: rows < 0, ld < 4, ld % 4, n_slots < 1, reqs/max_blocks/block_size
 *         < 1, null pointers, misalignment -> INVALID_ARG; S not in [1, 64],
 *         I < 1, block_size not 16, 32 or a multiple of 64, sizes past the
 *         32-bit tensor coordinates -> UNSUPPORTED; tensor-map encoding or
 *         launch failure -> CUDA.
 */
dsa_status dsa_indexer_logits(const uint8_t* q, const float* weights, const uint8_t* k_cache,
                              int64_t n_slots, const int32_t* block_table, int reqs,
                              int max_blocks, int block_size, const int32_t* row_to_req,
                              const int32_t* row_starts, const int32_t* row_ends, int rows,
                              int S, int I, float* logits, int64_t ld, uint32_t* err_flags,
                              cudaStream_t stream);

/*
 * dsa_fused_norm_rope - the cache rows of new tokens for the PCP prefill path.
 * PR #52046 report, "DSV3.2 PCP sharding": sections 功能与动机 (PCP shards the
 * sequence while the KV cache is replicated, so new cache rows are gathered
 * before they are inserted) and 实现拆解 item 1 / 关键源码片段
 * (`_fused_norm_rope_kernel`, pid == 1: RMS norm of kv_c, interleaved RoPE of
 * k_pe, results materialised to output buffers and/or written into the cache
 * at the token's slot).
 *
 * For token t (position p = positions[t]):
 *   kv_out[t]  = kv_c[t] / sqrt(mean(kv_c[t]^2) + eps) * norm_weight
 *   kpe_out[t] = k_pe[t] with each pair (2i, 2i+1) rotated: (x1 c - x2 s,
 *                x2 c + x1 s), c = cos_sin_cache[p][i], s = cos_sin_cache[p][32 + i]
 * computed in fp32 from bf16 inputs, stored as bf16 (round to nearest even).
 *
 *   kv_c, kv_out   [T][DSA_MLA_DV] bf16 (uint16 bit patterns), 16-byte aligned
 *   k_pe, kpe_out  [T][DSA_MLA_DQK - DSA_MLA_DV] bf16, 4-byte aligned
 *   positions      [T] int32; norm_weight [DSA_MLA_DV] fp32, 16-byte aligned
 *   cos_sin_cache  [max_pos][64] fp32: 32 cosines then 32 sines per position
 *   kv_out/kpe_out both or neither (materialise for the PCP gather);
 *   slot_mapping [T] int32 and kv_cache [n_slots][DSA_MLA_DQK] bf16 (16-byte
 *   aligned) both or neither: row slot_mapping[t] of the cache receives kv_out
 *   then kpe_out (a slot < 0 writes nothing).  At least one of the two modes.
 *   err_flags  DSA_FLAG_BOUNDS if a position is outside [0, max_pos) (that
 *              token's k_pe is not rotated) or a slot is >= n_slots (skipped).
 * Errors: T < 0, max_pos < 1, eps negative or not finite, an output pair half
 *         given, no output, null pointers, misalignment -> INVALID_ARG.
 */
dsa_status dsa_fused_norm_rope(const uint16_t* kv_c, const uint16_t* k_pe,
                               const int32_t* positions, const float* norm_weight, float eps,
                               const float* cos_sin_cache, int max_pos, int T, uint16_t* kv_out,
                               uint16_t* kpe_out, const int32_t* slot_mapping, uint16_t* kv_cache,
                               int64_t n_slots, uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_kv_cache_insert - gathered cache rows into the paged KV cache.
 * PR #52046 report, "DSV3.2 PCP sharding", section 实现拆解 item 3
 * (`maybe_gather_mla_latent_cache_inputs` gathers the PCP ranks' materialised
 * rows, then `do_kv_cache_update` inserts them).  With the ranks' slices held
 * in one buffer in rank order (the gather of contiguous sequence slices is
 * their concatenation), row t goes to slot slot_mapping[t]:
 *   kv_cache[slot][0 .. DSA_MLA_DV) = kv_rows[t], then kpe_rows[t].
 *   kv_rows [T][DSA_MLA_DV] bf16, 16-byte aligned; kpe_rows [T][64] bf16,
 *   4-byte aligned; kv_cache [n_slots][DSA_MLA_DQK] bf16, 16-byte aligned.
 *   err_flags  DSA_FLAG_BOUNDS if a slot is >= n_slots (skipped); slots < 0
 *              write nothing.
 * Errors: T < 0, n_slots < 1, null pointers, misalignment -> INVALID_ARG.
 */
dsa_status dsa_kv_cache_insert(const uint16_t* kv_rows, const uint16_t* kpe_rows,
                               const int32_t* slot_mapping, int T, uint16_t* kv_cache,
                               int64_t n_slots, uint32_t* err_flags, cudaStream_t stream);

/*
 * dsa_indexer_steps_noalloc - dsa_shard_topk_pack, dsa_merge_topk_stable and
 * dsa_convert_index_compact in turn, with the packed candidates held in a
 * static device array of this library (DSA_NOALLOC_SCRATCH_BYTES) instead of a
 * caller buffer.  No counterpart on the pages: a convenience for callers that
 * cannot allocate the [rows][S*K][2] candidate buffer.
 *
 * Arguments as the three entry points it calls (ids [rows][K] is the merge's
 * output and the convert's input; scores and local_idx are not produced).
 * It enqueues three kernels on `stream`.  Calls on one device share the array:
 * they must not overlap in time.  The array's address is looked up in the
 * current context on every call.
 * Errors: rows * S * K * 8 > DSA_NOALLOC_SCRATCH_BYTES -> UNSUPPORTED; then
 *         every argument check of the three entry points, before anything is
 *         enqueued (the first that fails is returned and nothing is touched);
 *         the array's address cannot be looked up -> CUDA.
 */
dsa_status dsa_indexer_steps_noalloc(const float* logits, int64_t ld, int rows, int S, int I,
                                     int K, const int32_t* row_starts, const int32_t* row_ends,
                                     const int32_t* block_table, int reqs, int max_blocks,
                                     int block_size, const int32_t* row_to_req, int32_t* ids,
                                     int32_t* slots, int32_t* counts, uint32_t* err_flags,
                                     cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
