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
// One CTA per (row, shard, group of 128 heads, half of the 512 output
// dimensions); the two halves are adjacent in the grid, run side by side and
// share the gathered rows in L2.  Fifth-generation tensor cores, warp-
// specialised, tiles of 64 selected tokens:
//  * the group's query (128 heads x 576 bf16) stays on chip for the whole slot
//    list: its first 320 dimensions in tensor memory (written once by the
//    softmax warps, a head per lane), the other 256 in shared memory (four
//    64-column blocks, 128-byte swizzle, K-major, one TMA tensor copy each);
//  * warps 0-3 gather the selected cache rows, two warps per stage (32 rows
//    of a tile each), tiles alternating between the stages: 16-byte
//    asynchronous copies (cp.async, eight lanes per 128-byte row segment)
//    placed in the 128-byte-swizzled layout, nine 64-column blocks of
//    [64 tokens x 64 bf16]; a warp waits for its own copies, makes them
//    visible to the tensor cores' proxy and arrives;
//  * one thread of warp 4 issues the MMAs: S = Q K^T as 36 tcgen05.mma
//    kind::f16 (M = 128 heads, N = 64 tokens, K = 16; bf16 in, fp32 out; A
//    from tensor memory for the first 20 steps, from shared memory for the
//    rest), and O += P V as four MMAs (N = 256 output dimensions, K = 16
//    tokens; A = P from tensor memory, B = this half's four value blocks of the
//    same gathered tile read MN-major); it polls both and issues S of tile
//    t + 1 or P V of tile t, whichever is ready first, so the softmax of a
//    tile overlaps the tensor work and a stage is freed as early as possible;
//  * warps 5-8, a thread per head (its tensor-memory lane), run the softmax
//    in the exp2 domain: scores out of tensor memory, masked tokens to -inf,
//    weights relative to a reference maximum that moves only when a tile's
//    maximum exceeds it by more than 8 (so O in tensor memory is rescaled
//    rarely), bf16 weights back into tensor memory as the A operand of P V;
//    they also write the outputs.
// An MMA of M = 128 and K = 16 takes about 50 cycles on this GPU whatever its
// N up to 64 (and N / 2 cycles above 128), so the scores' N is as large as
// the on-chip memory allows: tensor memory holds O (256 columns), S (64), P
// (32) and the query's first 320 dimensions (160); shared memory two stages of
// 72 KB and 64 KB of the query.
// Two row sums are kept: of the fp32 weights (the LSE) and of the bf16-rounded
// weights that enter P V (O's normaliser).  Every wait is bounded; a wait that
// runs out raises DSA_FLAG_TIMEOUT and stops the CTA's roles, which drain
// their copies and MMAs in flight before the tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kDqk = DSA_MLA_DQK;            // 576: latent 512 + rope 64
constexpr int kDv = DSA_MLA_DV;              // 512
constexpr int kHeads = 128;                  // heads per CTA: the MMA's M
constexpr int kHalf = kDv / 2;               // output dimensions per CTA
constexpr int kTile = 64;                    // tokens per tile: the scores' N
constexpr int kStages = 2;                   // tiles in flight
constexpr int kBlocks = kDqk / 64;           // 9 column blocks of 64 bf16 (128 bytes)
constexpr int kQtBlocks = 5;                 // query blocks held in tensor memory
constexpr int kQsBlocks = kBlocks - kQtBlocks;   // and in shared memory
constexpr int kQBlock = kHeads * 128;        // bytes of one query block
constexpr int kKvBlock = kTile * 128;        // bytes of one tile block
constexpr int kVBlocks = kHalf / 64;         // 4 value blocks per half
constexpr int kGatherWarps = 4;              // two per stage, 32 rows of a tile each
constexpr int kABlocks = kBlocks - kVBlocks; // 5 blocks only the scores read
constexpr int kMmaWarp = kGatherWarps;
constexpr int kSoftmaxWarps = 4;
constexpr int kThreads = (kGatherWarps + 1 + kSoftmaxWarps) * 32;
// Tensor-memory columns (fp32 or packed bf16 pairs, a head per lane).
constexpr int kOCol = 0;                     // O: 256
constexpr int kSCol = 256;                   // S: 64
constexpr int kPCol = 320;                   // P: 64 tokens as 32 bf16 pairs
constexpr int kQCol = 352;                   // query dimensions 0..319: 160
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleGap = 8.f;           // weights stay below 2^8 before a rescale
#ifdef DSA_TEST_STALLED_COPY
// The test-only build (never libdsa.so): every stage's part-A barrier expects
// one arrival that nothing makes, so the first scores' wait runs out (every
// copy still lands) and the kernel returns with DSA_FLAG_TIMEOUT.
constexpr uint32_t kStalledArrivals = 1;
#else
constexpr uint32_t kStalledArrivals = 0;
#endif

static_assert(kGatherWarps == 2 * kStages, "two gathering warps per stage");
static_assert(kBlocks * 64 == kDqk && kVBlocks * 64 == kHalf, "column blocks");
static_assert(kQCol + kQtBlocks * 32 == kTmemCols && kPCol + kTile / 2 == kQCol &&
                  kSCol + kTile == kPCol && kOCol + kHalf == kSCol,
              "tensor-memory columns");

struct alignas(1024) MlaSmem {
  uint8_t kv[kStages][kBlocks][kKvBlock];    // 147456: gathered tiles
  uint8_t q[kQsBlocks][kQBlock];             // 65536: query dimensions 320..575
  uint32_t vmask[4][2];                      // valid tokens of tile t, at t & 3
  // A stage in two parts: the five blocks only the scores read (A) and this
  // half's four value blocks (B), filled and freed separately.
  uint64_t qfull, qtm, fullA[kStages], fullB[kStages], emptyA[kStages], emptyB[kStages];
  uint64_t sfull, sfree, pfull, pvdone, drain;
  uint32_t tmem;
  int abort;
};

struct MlaArgs {
  const __nv_bfloat16* q;        // [rows][H][kDqk]
  const __nv_bfloat16* cache;    // [S][n_slots][kDqk]
  const int32_t* slots;          // [S][rows][K]
  const int32_t* counts;         // [S][rows]
  int64_t n_slots;
  int rows, H, K, hgroups, box_h;
  float c2;                      // scale * log2(e)
  __nv_bfloat16* out;            // [S][rows][H][kDv]
  float* lse2;                   // [S][rows][H]
  uint32_t* flags;
};

// Column block of step i of part A (the blocks only the scores read) and of
// part B (this half's value blocks): half 0 reads values from blocks 0-3, so
// its part A is 4-8; half 1 reads 4-7, so its part A is 0-3 and 8.
__host__ __device__ constexpr int block_a(int half, int i) {
  return half == 0 ? kVBlocks + i : (i < kVBlocks ? i : kBlocks - 1);
}
__host__ __device__ constexpr int block_b(int half, int i) { return half * kVBlocks + i; }

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (bits 16-29), stride byte offset >> 4 (bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode (bits 61-63: 2 = 128-byte,
// the layout TMA and the gathers write).  K-major operands: the stride is that of 8-row
// groups, the leading offset unused (1).  MN-major 128-byte swizzle: the
// leading offset steps between 64-element atoms along N, the stride between
// 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)swizzle << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A
// and B bf16 (bits 7-9, 10-12 = 1), A K-major, B K-major or MN-major (bit 16),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
constexpr uint32_t idesc_bf16(int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kHeads >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_tc(uint32_t d_tmem, uint64_t a, uint64_t b,
                                            uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

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

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// The same MMA with A (M x 16 bf16, a row per lane as 8 columns of packed
// pairs) in tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void cp_async16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.  The
// wait is followed by empty statements naming every destination register as
// read and written, so no use of them can be scheduled before it.
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
#define DSA_TMEM_ST16(o)                                                                    \
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, " \
               "%8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr + (uint32_t)(o)),  \
               "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]),   \
               "r"(r[o + 5]), "r"(r[o + 6]), "r"(r[o + 7]), "r"(r[o + 8]), "r"(r[o + 9]),   \
               "r"(r[o + 10]), "r"(r[o + 11]), "r"(r[o + 12]), "r"(r[o + 13]),              \
               "r"(r[o + 14]), "r"(r[o + 15])                                               \
               : "memory")

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  DSA_TMEM_LD16(0);
  DSA_TMEM_LD16(16);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  DSA_WAIT_LD16(0);
  DSA_WAIT_LD16(16);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  DSA_TMEM_ST16(0);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  DSA_TMEM_ST16(0);
  DSA_TMEM_ST16(16);
}
#undef DSA_TMEM_LD16
#undef DSA_WAIT_LD16
#undef DSA_TMEM_ST16

__device__ __forceinline__ bool aborted(const MlaSmem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

// Bounded wait that also gives up once another role of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(MlaSmem& sm, uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (aborted(sm)) return false;
    if (i > 64) __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ void abort_cta(MlaSmem& sm, uint32_t* flags) {
  raise_flag(flags, DSA_FLAG_TIMEOUT);
  *reinterpret_cast<volatile int*>(&sm.abort) = 1;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// 2^x (ex2.approx.ftz.f32: relative error about 2^-22, results below 2^-126
// flushed to zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fused multiply-adds in one instruction (fma.rn.f32x2) and two additions
// (add.rn.f32x2), each rounded as the scalar operation would be.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}


// ---- warps 0-3: the query's shared-memory blocks, then the tiles' rows -----
// Warps w and w + 2 gather tiles w, w + 2, ... (w = 0, 1) into stage w, rows
// 0-31 and 32-63 of each.  Lane l owns one token of those rows (slot,
// validity); the copies go four rows at a time, eight lanes per row segment
// of one 64-column block (128 bytes read contiguously).  Part A of a tile
// goes as soon as the scores of the stage's previous tile are done, part B
// once its P V is.
__device__ __forceinline__ void copy_part(const MlaArgs& a, uint32_t stage, int64_t row_base,
                                          int y, int half, bool part_a) {
  const int lane = threadIdx.x & 31;
  const int cc = lane & 7, rsub = lane >> 3;
#pragma unroll 2
  for (int rq = 0; rq < 8; ++rq) {
    const int jr = 4 * rq + rsub;                      // row among this warp's 32
    const int yj = __shfl_sync(kFull, y, jr);
    const char* src = reinterpret_cast<const char*>(a.cache + (row_base + yj) * kDqk) + cc * 16;
    // The row's swizzle phase within its 8-row group is jr & 7.
    const uint32_t dst = stage + (uint32_t)(jr * 128 + ((cc ^ (jr & 7)) << 4));
    if (part_a) {
#pragma unroll
      for (int i = 0; i < kABlocks; ++i) {
        const int kb = block_a(half, i);
        cp_async16_cg(dst + kb * kKvBlock, src + kb * 128);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kVBlocks; ++i) {
        const int kb = block_b(half, i);
        cp_async16_cg(dst + kb * kKvBlock, src + kb * 128);
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // This lane's copies (generic proxy) before the MMAs read them (async proxy).
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void gather_tiles(const MlaArgs& a, MlaSmem& sm,
                                             const CUtensorMap* tm_q, int r, int hg, int half,
                                             int64_t row_base, int count, int ntiles,
                                             const int32_t* slot_row) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int st = warp % kStages, part = warp / kStages;   // stage, 32-row half of the tile
  if (warp == 0 && lane == 0) {
    mbar_expect_tx(&sm.qfull, (uint32_t)(kQsBlocks * a.box_h * 128));
    for (int i = 0; i < kQsBlocks; ++i)
      tma_load_3d(sm.q[i], tm_q, (kQtBlocks + i) * 64, hg * kHeads, r, &sm.qfull);
  }
  const uint32_t stage = smem_u32(sm.kv[st][0]) + (uint32_t)(part * 32 * 128);
  bool bad = false, ok = true;
  for (int t = st, k = 0; t < ntiles; t += kStages, ++k) {
    if (k >= 1) ok = wait_or_abort(sm, &sm.emptyA[st], (uint32_t)(k - 1) & 1u);
    if (!__all_sync(kFull, ok)) break;
    const int j = t * kTile + part * 32 + lane;
    const int slot = j < count ? __ldg(slot_row + j) : -1;
    const bool in = slot >= 0 && (int64_t)slot < a.n_slots;
    bad |= j < count && !in;
    const unsigned v = __ballot_sync(kFull, in);
    // A token left out reads a row the tile already reads (its weight is 0),
    // or the shard's first row when these 32 tokens have no valid one.
    const int sub = v ? __shfl_sync(kFull, slot, __ffs(v) - 1) : 0;
    const int y = in ? slot : sub;
    if (lane == 0) sm.vmask[t & 3][part] = v;   // published by this lane's arrivals
    copy_part(a, stage, row_base, y, half, true);
    mbar_arrive1(&sm.fullA[st]);
    if (k >= 1) ok = wait_or_abort(sm, &sm.emptyB[st], (uint32_t)(k - 1) & 1u);
    if (!__all_sync(kFull, ok)) break;
    copy_part(a, stage, row_base, y, half, false);
    mbar_arrive1(&sm.fullB[st]);
  }
  if (!__all_sync(kFull, ok) && lane == 0 && !aborted(sm)) abort_cta(sm, a.flags);
  if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  // The query's copies land before this warp, and so the CTA, exits.
  if (warp == 0 && lane == 0 && !mbar_wait(&sm.qfull, 0)) abort_cta(sm, a.flags);
}

// ---- warp 4, one thread: the MMAs ------------------------------------------
// Scores in two parts following the stage's (part A's five blocks, then part
// B's four), P V, each issued as soon as its operands are ready: P V of tile
// t first (it frees part B of the stage), then part B of S, then part A of
// the next S once the softmax has read the previous scores.
template <int HALF>
__device__ __forceinline__ void issue_mmas(const MlaArgs& a, MlaSmem& sm, uint32_t tmem,
                                           int ntiles) {
  constexpr uint32_t kIdS = idesc_bf16(kTile, false);
  constexpr uint32_t kIdO = idesc_bf16(kHalf, true);
  bool ok = wait_or_abort(sm, &sm.qfull, 0) && wait_or_abort(sm, &sm.qtm, 0);
  tc_fence_after();
  const uint64_t qd = smem_desc(smem_u32(sm.q[0]), 16, 1024, 2);
  const uint32_t d_s = tmem + kSCol, d_o = tmem + kOCol, a_q = tmem + kQCol, a_p = tmem + kPCol;
  // The four K-steps of one 64-column block kb (descriptors advance by bytes
  // >> 4: 16 K-elements = 32 bytes = 2, one block = its size >> 4); A is the
  // query block, in tensor memory for kb < kQtBlocks.
  auto block_steps = [&](uint64_t kd, int kb, bool first) {
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const uint64_t db = kd + (uint64_t)(kb * (kKvBlock >> 4) + k4 * 2);
      const uint32_t acc = (first && k4 == 0) ? 0u : 1u;
      if (kb < kQtBlocks)
        mma_bf16_ts(d_s, a_q + (uint32_t)(kb * 32 + k4 * 8), db, kIdS, acc);
      else
        mma_bf16_tc(d_s, qd + (uint64_t)((kb - kQtBlocks) * (kQBlock >> 4) + k4 * 2), db, kIdS,
                    acc);
    }
  };
  int na = 0, nb = 0;                        // S parts A and B issued so far
  uint32_t idle = 0;                         // polls since the last issue
  for (int t = 0; ok && t < ntiles;) {
    if (nb > t && mbar_test(&sm.pfull, (uint32_t)t & 1u)) {
      tc_fence_after();
      // V: this half's four blocks, MN-major: 64-column atoms kKvBlock apart,
      // 8-token groups 1024 bytes apart; 16 tokens a step = 2048 bytes.
      const uint64_t vd = smem_desc(smem_u32(sm.kv[t & 1][HALF * kVBlocks]), kKvBlock, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16_ts(d_o, a_p + (uint32_t)(kk * 8), vd + (uint64_t)(kk * (2048 >> 4)), kIdO,
                    (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&sm.emptyB[t & 1]);
      mma_commit(&sm.pvdone);
      ++t;
      idle = 0;
      continue;
    }
    if (na > nb && mbar_test(&sm.fullB[nb & 1], (uint32_t)(nb >> 1) & 1u)) {
      tc_fence_after();
      const uint64_t kd = smem_desc(smem_u32(sm.kv[nb & 1][0]), 16, 1024, 2);
#pragma unroll
      for (int i = 0; i < kVBlocks; ++i) block_steps(kd, block_b(HALF, i), false);
      mma_commit(&sm.sfull);
      mma_commit(&sm.emptyA[nb & 1]);
      ++nb;
      idle = 0;
      continue;
    }
    if (na == nb && na < ntiles && mbar_test(&sm.fullA[na & 1], (uint32_t)(na >> 1) & 1u) &&
        (na == 0 || mbar_test(&sm.sfree, (uint32_t)(na - 1) & 1u))) {
      tc_fence_after();
      const uint64_t kd = smem_desc(smem_u32(sm.kv[na & 1][0]), 16, 1024, 2);
#pragma unroll
      for (int i = 0; i < kABlocks; ++i) block_steps(kd, block_a(HALF, i), i == 0);
      ++na;
      idle = 0;
      continue;
    }
    // Nothing ready: poll again (bounded, as every wait).
    if (++idle >= 4 * kWaitPolls || aborted(sm)) {
      ok = false;
      break;
    }
    if (idle > 64) __nanosleep(32);
  }
  if (!ok && !aborted(sm)) abort_cta(sm, a.flags);
  // Every MMA issued completes before the tensor memory is freed.
  mma_commit(&sm.drain);
  if (!mbar_wait(&sm.drain, 0)) abort_cta(sm, a.flags);
}

// ---- warps 5-8: the query's tensor-memory part, softmax, the outputs -------
__device__ __forceinline__ void softmax_and_store(const MlaArgs& a, MlaSmem& sm, uint32_t tmem,
                                                  int r, int half, int ntiles, int64_t head0,
                                                  int hg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int quad = warp & 3;                 // the tensor-memory lanes this warp may access
  const int h = quad * 32 + lane;            // this thread's head within the group
  const int gh = hg * kHeads + h;
  const bool active = gh < a.H;
  const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);

  // Query dimensions 0..319 of this head into tensor memory (zeros past H),
  // in two batches of 20 loads in flight.
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.q + ((int64_t)r * a.H + gh) * kDqk);
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      uint4 x[20];
#pragma unroll
      for (int i = 0; i < 20; ++i) x[i] = active ? __ldg(src + b * 20 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 80; c += 16) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] = x[c / 4 + i].x;
          v[4 * i + 1] = x[c / 4 + i].y;
          v[4 * i + 2] = x[c / 4 + i].z;
          v[4 * i + 3] = x[c / 4 + i].w;
        }
        tmem_st16(trow + (uint32_t)(kQCol + b * 80 + c), v);
      }
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive1(&sm.qtm);
  }

  float m = -INFINITY, l = 0.f, w = 0.f;
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int st = t & 1;
    // Part B of the tile has landed: its validity masks are visible.
    ok = wait_or_abort(sm, &sm.sfull, (uint32_t)t & 1u) &&
         wait_or_abort(sm, &sm.fullB[st], (uint32_t)(t >> 1) & 1u);
    if (!__all_sync(kFull, ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(trow + kSCol, r0);
    tmem_ld32(trow + kSCol + 32, r1);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive1(&sm.sfree);
    const uint32_t vm0 = sm.vmask[t & 3][0], vm1 = sm.vmask[t & 3][1];
    // Every token valid and a positive scale (the usual case, the same for the
    // whole CTA): the maximum of the raw scores, scaled once, in four
    // independent chains; otherwise masked tokens are -inf.
    const bool full = (vm0 & vm1) == kFull && a.c2 > 0.f;
    float mx;
    if (full) {
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 32; ++j)
        m4[j & 3] = fmaxf(m4[j & 3], fmaxf(__uint_as_float(r0[j]), __uint_as_float(r1[j])));
      mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.c2;
    } else {
      mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if ((vm0 >> j) & 1u) mx = fmaxf(mx, __uint_as_float(r0[j]) * a.c2);
        if ((vm1 >> j) & 1u) mx = fmaxf(mx, __uint_as_float(r1[j]) * a.c2);
      }
    }
    const float mn = mx > m + kRescaleGap ? mx : m;   // m = -inf takes any finite max
    const float alpha = m == -INFINITY ? 1.f : fast_exp2(m - mn);
    const float ref = mn == -INFINITY ? 0.f : mn;
    // Weights 2^(s c2 - ref) two at a time (one fused multiply-add pair), packed
    // to bf16; the fp32 and the bf16-rounded sums in two-wide accumulators.
    uint32_t pk[kTile / 2];
    float2 as[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float2 ab[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    const float2 c2v = make_float2(a.c2, a.c2), nref = make_float2(-ref, -ref);
#pragma unroll
    for (int j = 0; j < kTile / 2; ++j) {
      const uint32_t* rr = j < 16 ? r0 : r1;
      const int i = 2 * (j & 15);
      float2 xv = ffma2(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])), c2v, nref);
      if (!full) {
        const uint32_t vm = j < 16 ? vm0 : vm1;
        if (!((vm >> i) & 1u)) xv.x = -INFINITY;
        if (!((vm >> (i + 1)) & 1u)) xv.y = -INFINITY;
      }
      const float e0 = fast_exp2(xv.x), e1 = fast_exp2(xv.y);
      pk[j] = pack_bf16(e0, e1);
      as[j & 1] = fadd2(as[j & 1], make_float2(e0, e1));
      ab[j & 1] = fadd2(ab[j & 1], make_float2(__uint_as_float(pk[j] << 16),
                                               __uint_as_float(pk[j] & 0xFFFF0000u)));
    }
    const float s = (as[0].x + as[0].y) + (as[1].x + as[1].y);
    const float sb = (ab[0].x + ab[0].y) + (ab[1].x + ab[1].y);
    l = l * alpha + s;
    w = w * alpha + sb;
    m = mn;
    // P V of the previous tile is done: the weights' columns are free and O
    // holds every earlier tile.
    if (t > 0) ok = wait_or_abort(sm, &sm.pvdone, (uint32_t)(t - 1) & 1u);
    if (!__all_sync(kFull, ok)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (__any_sync(kFull, alpha != 1.f)) {     // the reference moved: rescale O
#pragma unroll 1
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o[32];
        tmem_ld32(trow + (uint32_t)(kOCol + c), o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
        tmem_st32(trow + (uint32_t)(kOCol + c), o);
      }
    }
    tmem_st32(trow + kPCol, pk);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive1(&sm.pfull);
  }
  if (ok && ntiles > 0) ok = wait_or_abort(sm, &sm.pvdone, (uint32_t)(ntiles - 1) & 1u);
  if (!__all_sync(kFull, ok)) {
    if (lane == 0 && !aborted(sm)) abort_cta(sm, a.flags);
    return;
  }
  tc_fence_after();
  // O / w in bf16 (this CTA's 256 dimensions); lse2 = m + log2 l.
  const float inv = w > 0.f ? 1.f / w : 0.f;
  __nv_bfloat16* orow = a.out + (head0 + h) * kDv + half * kHalf;
#pragma unroll 1
  for (int c = 0; c < kHalf; c += 32) {
    uint32_t o[32];
    tmem_ld32(trow + (uint32_t)(kOCol + c), o);
    if (active) {
      uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint32_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          b[i] = pack_bf16(__uint_as_float(o[8 * v + 2 * i]) * inv,
                           __uint_as_float(o[8 * v + 2 * i + 1]) * inv);
        dst[v] = make_uint4(b[0], b[1], b[2], b[3]);
      }
    }
  }
  if (active && half == 0) a.lse2[head0 + h] = l > 0.f ? m + log2f(l) : -INFINITY;
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const MlaArgs a) {
  extern __shared__ unsigned char mla_smem_raw[];
  MlaSmem& sm = *reinterpret_cast<MlaSmem*>(
      (reinterpret_cast<uintptr_t>(mla_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  const int half = blockIdx.x & 1;
  const int x = blockIdx.x >> 1;
  const int hg = x % a.hgroups;
  const int pair = x / a.hgroups;            // s * rows + r
  const int s = pair / a.rows, r = pair - s * a.rows;
  int count = __ldg(a.counts + pair);
  if ((count < 0 || count > a.K) && tid == 0 && half == 0) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  count = min(max(count, 0), a.K);
  const int ntiles = (count + kTile - 1) / kTile;
  const int64_t head0 = (int64_t)pair * a.H + hg * kHeads;   // first head of the group
  const int nheads = min(kHeads, a.H - hg * kHeads);

  if (count == 0) {
    // Nothing selected on this shard: O = 0, lse2 = -inf.
    for (int i = tid; i < nheads * (kHalf / 8); i += kThreads)
      *reinterpret_cast<uint4*>(a.out + (head0 + i / (kHalf / 8)) * kDv + half * kHalf +
                                (i % (kHalf / 8)) * 8) = make_uint4(0, 0, 0, 0);
    if (half == 0 && tid < nheads) a.lse2[head0 + tid] = -INFINITY;
    return;
  }

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(&sm.qfull, 1);
    mbar_init(&sm.qtm, kSoftmaxWarps);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.fullA[i], 32 * kGatherWarps / kStages + kStalledArrivals);   // every gathering lane
      mbar_init(&sm.fullB[i], 32 * kGatherWarps / kStages);
      mbar_init(&sm.emptyA[i], 1);
      mbar_init(&sm.emptyB[i], 1);
    }
    mbar_init(&sm.sfull, 1);
    mbar_init(&sm.sfree, kSoftmaxWarps);
    mbar_init(&sm.pfull, kSoftmaxWarps);
    mbar_init(&sm.pvdone, 1);
    mbar_init(&sm.drain, 1);
    sm.abort = 0;
    mbar_init_fence();
  }
  if (a.box_h < kHeads && warp > kMmaWarp) {
    // Fewer heads than a box: the shared-memory query rows past them are zeros.
    const int per_block = (kHeads - a.box_h) * 8;   // 16-byte chunks
    for (int i = tid - (kMmaWarp + 1) * 32; i < kQsBlocks * per_block; i += kSoftmaxWarps * 32)
      *reinterpret_cast<uint4*>(sm.q[i / per_block] + a.box_h * 128 + (i % per_block) * 16) =
          make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp < kGatherWarps) {
    gather_tiles(a, sm, &tm_q, r, hg, half, (int64_t)s * a.n_slots, count, ntiles,
                 a.slots + (int64_t)pair * a.K);
  } else if (warp == kMmaWarp) {
    if ((tid & 31) == 0) {
      if (half == 0) issue_mmas<0>(a, sm, tmem, ntiles);
      else issue_mmas<1>(a, sm, tmem, ntiles);
    }
    __syncwarp();
  } else {
    softmax_and_store(a, sm, tmem, r, half, ntiles, head0, hg);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

// The queries as [rows][H] rows of kDqk bf16: boxes of 64 columns (128 bytes,
// 128-byte swizzle) by box_h heads of one row.
bool encode_queries(CUtensorMap* map, const void* q, int rows, int H, int box_h) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kDqk, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kDqk * 2, (cuuint64_t)kDqk * 2 * (cuuint64_t)H};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_h, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

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
  if (S < 1 || S > DSA_MAX_SHARDS || H < 64 || H % 64) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!q || !kv_cache || !slots || !counts || !out || !lse2) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
  if (n_slots > (int64_t)INT32_MAX + 1) return DSA_ERR_UNSUPPORTED;
  const int hgroups = (H + kHeads - 1) / kHeads;
  const int64_t blocks = (int64_t)rows * S * hgroups * 2;
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  const int box_h = H < kHeads ? H : kHeads;
  CUtensorMap tm_q;
  if (!encode_queries(&tm_q, q, rows, H, box_h)) return DSA_ERR_CUDA;
  const int smem = (int)sizeof(MlaSmem) + 1024;
  if (cudaFuncSetAttribute(sparse_mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return DSA_ERR_CUDA;
  const MlaArgs a{reinterpret_cast<const __nv_bfloat16*>(q),
                  reinterpret_cast<const __nv_bfloat16*>(kv_cache),
                  slots,
                  counts,
                  n_slots,
                  rows,
                  H,
                  K,
                  hgroups,
                  box_h,
                  scale * kLog2e,
                  reinterpret_cast<__nv_bfloat16*>(out),
                  lse2,
                  err_flags};
  const cudaError_t e = launch_kernel(sparse_mla_decode_kernel, dim3((unsigned)blocks),
                                      dim3(kThreads), (size_t)smem, stream, 0, tm_q, a);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
