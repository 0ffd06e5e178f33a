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
// Persistent CTAs walk work items (shard, group of G rows, chunk of 16 tiles
// of 128 local slots) round-robin.  G = 4 when every row reads the same
// request (one key tile then serves four rows), else 1.  Warp roles:
//   producer (warp E)  TMA: per item the group's query heads (G x 8 KB) and
//            weights into one of two slots, per tile the 128 keys, one 2-D
//            tensor copy per block of the paged cache (a 64-row box for
//            64-token blocks), into a 4-stage ring, 128-byte swizzle.  It also
//            allocates and frees the tensor memory.
//   MMA (warp E + 1, one thread)  per tile D[128 tokens][G x 64 heads] =
//            K_tile . Q^T: four tcgen05.mma kind::f8f6f4 (N = 64 G, K = 32
//            each) into the next accumulator in tensor memory; commits free
//            the key stage, hand the accumulator to the epilogue and, after an
//            item's last tile, free its query slot.
//   epilogue (warps 0 .. E-1, E = 4 G)  warp e reads tensor-memory lanes
//            32 (e % 4) .. + 31 (one token per thread) of row e / 4, applies
//            ReLU and the head weights (read from shared memory) and stores
//            one logit (a warp writes 32 consecutive slots); then it releases
//            the accumulator.  Four accumulators when ungrouped (two CTAs per
//            SM), two when grouped: the MMAs run ahead of the epilogue.
// Barrier phases run on across items (a tile counter and an item counter).
// Every wait is bounded: a wait that runs out raises DSA_FLAG_TIMEOUT, the
// roles stop, drain their copies and MMAs (bounded) and the tensor memory is
// freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kHeads = DSA_IDX_HEADS;      // 64
constexpr int kDim = DSA_IDX_DIM;          // 128 fp8 values = 128 bytes per row
constexpr int kTile = 128;                 // tokens per tile = MMA M
constexpr int kTilesPerItem = 32;
// Block-table entries one item can need: 16 tiles of 128 slots in blocks of
// at least 16 slots, plus one for a range that starts mid-block.
constexpr int kItemBlocks = kTilesPerItem * 128 / 16 + 1;
constexpr uint32_t kTileBytes = kTile * kDim;
constexpr uint32_t kQBytes = kHeads * kDim;  // one row's query heads

template <int G, int P>
struct LogitsCfg {
  // G rows per MMA (N = 64 G), P passes of the MMAs over each key tile: an
  // item holds R = G P rows, and each key tile read from memory serves all R.
  static constexpr int R = G * P;
  // Key stages: enough bytes in flight to cover the latency of the key reads
  // at the rate the MMAs consume them (one CTA per SM when grouped).
  static constexpr int kStages = G == 1 ? 4 : 4;
  // One epilogue warp per (lane quarter, row of a pass): a tile's epilogue
  // latency is one row's, and the MMAs run ahead by as many accumulators as
  // the tensor memory holds (two CTAs per SM when ungrouped, one when grouped).
  static constexpr int kEpiWarps = 4 * G;
  static constexpr int kAccBufs = G == 1 ? 4 : 2;
  static constexpr int kThreads = (kEpiWarps + 2) * 32;
  static constexpr int kProducer = kEpiWarps, kMma = kEpiWarps + 1;
  static constexpr uint32_t kAccCols = (uint32_t)G * kHeads;   // one accumulator
  static constexpr uint32_t kTmemCols = kAccBufs * kAccCols;   // 256 or 512
};

template <int G, int P>
struct alignas(1024) LogitsSmem {
  static constexpr int kStages = LogitsCfg<G, P>::kStages;
  static constexpr int R = G * P;
  uint8_t k[kStages][kTileBytes];          // 1024-aligned: the swizzle atom
  uint8_t q[2][R * kQBytes];               // the item's query heads, two slots
  float w[2][R * kHeads];                  // and weights
  int32_t pblk[kItemBlocks];               // the item's block-table entries
  uint64_t full[kStages], empty[kStages], qfull[2], qfree[2];
  uint64_t accfull[LogitsCfg<G, P>::kAccBufs], accempty[LogitsCfg<G, P>::kAccBufs], drain;
  uint64_t stall;                          // the test-only build's wait that runs out
  uint32_t tmem;
  int abort;
};

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A and B e4m3 (format 0), both K-major, N (bits 17-22: N >> 3), M = 128
// (bits 24-28: M >> 4).
constexpr uint32_t idesc_f8(int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTile >> 4) << 24);
}

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

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
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

// 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes (two
// 16-column loads, then one wait).  The wait is followed by empty statements
// that name every destination register as read and written, so no use of
// them can be scheduled before it.
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

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  DSA_TMEM_LD16(0);
  DSA_TMEM_LD16(16);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  DSA_WAIT_LD16(0);
  DSA_WAIT_LD16(16);
}
#undef DSA_TMEM_LD16
#undef DSA_WAIT_LD16

// Two fused multiply-adds in one instruction (fma.rn.f32x2): (a.x b.x + c.x,
// a.y b.y + c.y), each rounded as fmaf would.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}

template <typename Smem>
__device__ __forceinline__ bool aborted(const Smem& sm) {
  return *reinterpret_cast<const volatile int*>(&sm.abort) != 0;
}

// One work item: shard s, rows r0 .. r0 + nrows - 1 (nrows <= R), the tiles
// [t_lo, t_lo + ntiles) of local slots covering their ranges inside chunk c.
// Every role computes it the same way from the same inputs.
template <int R>
struct Item {
  int s, r0, nrows, ntiles;
  int64_t t_lo;
  int64_t lo[R], hi[R];
};

template <int R>
__device__ __forceinline__ Item<R> make_item(int it, int rows, int groups, int chunks,
                                             const int32_t* row_starts, const int32_t* row_ends,
                                             int64_t ld, const ShardMath& sh, bool* bad) {
  Item<R> x;
  const int c = it % chunks;
  const int sg = it / chunks;
  x.s = sg / groups;
  x.r0 = (sg - x.s * groups) * R;
  x.nrows = min(R, rows - x.r0);
  int64_t glo = INT64_MAX, ghi = 0;
#pragma unroll
  for (int g = 0; g < R; ++g) {
    x.lo[g] = x.hi[g] = 0;
    if (g < x.nrows) {
      const int r = x.r0 + g;
      int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
      if (st < 0) { st = 0; *bad = true; }
      if (en < st) { en = st; *bad = true; }
      int64_t lo = sh.local_len((uint32_t)st, x.s), hi = sh.local_len((uint32_t)en, x.s);
      if (hi > ld) { hi = ld; *bad = true; }
      if (lo > hi) { lo = hi; *bad = true; }
      x.lo[g] = lo;
      x.hi[g] = hi;
      if (hi > lo) {
        glo = min(glo, lo);
        ghi = max(ghi, hi);
      }
    }
  }
  if (ghi <= 0 || glo >= ghi) {
    x.t_lo = 0;
    x.ntiles = 0;
    return x;
  }
  x.t_lo = max(glo / kTile, (int64_t)c * kTilesPerItem);
  const int64_t t_hi = min((ghi + kTile - 1) / kTile, (int64_t)(c + 1) * kTilesPerItem);
  x.ntiles = (int)max((int64_t)0, t_hi - x.t_lo);
  return x;
}

template <int G, int P>
__global__ void __launch_bounds__(LogitsCfg<G, P>::kThreads, G == 1 ? 2 : 1)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_q, const float* __restrict__ w,
                          const int32_t* __restrict__ block_table, int reqs, int max_blocks,
                          int block_size, int box_rows, int64_t n_slots,
                          const int32_t* __restrict__ row_to_req,
                          const int32_t* __restrict__ row_starts,
                          const int32_t* __restrict__ row_ends, int rows, int S, int64_t ld,
                          int chunks, int nitems, float* __restrict__ logits, uint32_t* flags,
                          const ShardMath sh, const FastDiv fbs) {
  using Cfg = LogitsCfg<G, P>;
  constexpr int kStages = Cfg::kStages;
  constexpr int R = Cfg::R;
  extern __shared__ unsigned char logits_smem_raw[];
  LogitsSmem<G, P>& sm = *reinterpret_cast<LogitsSmem<G, P>*>(
      (reinterpret_cast<uintptr_t>(logits_smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = (rows + R - 1) / R;

  if (warp == Cfg::kProducer) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem)),
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 32 * Cfg::kMma) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.qfull[b], 1);
      mbar_init(&sm.qfree[b], 1 + Cfg::kEpiWarps);   // the MMA commit + every epilogue warp
    }
    for (int b = 0; b < Cfg::kAccBufs; ++b) {
      mbar_init(&sm.accfull[b], 1);
      mbar_init(&sm.accempty[b], Cfg::kEpiWarps);
    }
    mbar_init(&sm.drain, 1);
    mbar_init(&sm.stall, 1);
    sm.abort = 0;
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  bool bad = false;

  if (warp == Cfg::kProducer) {
    // ---- producer: the warp stages each item's block-table entries in shared
    // memory (one coalesced load), lane 0 issues the copies -----------------
    const int oob_y = (int)((int64_t)S * n_slots);   // past the cache: zero fill
    const int boxes = box_rows == 64 ? 2 : (box_rows == 32 ? 4 : 8);   // per tile of 128 slots
    int gt = 0, icount = 0;
    for (int it = blockIdx.x; it < nitems && !aborted(sm); it += gridDim.x) {
      const Item<R> x = make_item<R>(it, rows, groups, chunks, row_starts, row_ends, ld, sh, &bad);
      if (x.ntiles == 0) continue;
      const int req = row_to_req ? row_to_req[x.r0] : x.r0;
      const bool req_ok = req >= 0 && req < reqs;
      if (!req_ok) bad = true;
      const int32_t* bt = block_table + ((int64_t)x.s * reqs + (req_ok ? req : 0)) * max_blocks;
      int64_t ghi = 0;
#pragma unroll
      for (int g = 0; g < R; ++g) ghi = max(ghi, x.hi[g]);
      // Local slots are below ld < 2^31: 32-bit maps (no 64-bit division).
      const uint32_t tok_lo = (uint32_t)(x.t_lo * kTile);
      const uint32_t tok_end = (uint32_t)min((x.t_lo + x.ntiles) * kTile, ghi);
      const int blk0 = (int)fdiv(tok_lo, fbs);
      const int blk_end = min(max_blocks, (int)fdiv(tok_end + (uint32_t)block_size - 1u, fbs));
      const int nblk = max(0, blk_end - blk0);   // <= kItemBlocks
      __syncwarp();                      // lane 0 is done with the previous item's entries
      for (int i = lane; i < nblk; i += 32) sm.pblk[i] = req_ok ? bt[blk0 + i] : -1;
      __syncwarp();
      if (lane == 0) {
        const int qb = icount & 1;
        if (icount >= 2 && !mbar_wait(&sm.qfree[qb], (uint32_t)((icount >> 1) - 1) & 1u)) {
          raise_flag(flags, DSA_FLAG_TIMEOUT);
          sm.abort = 1;
        } else {
          mbar_expect_tx(&sm.qfull[qb], (uint32_t)R * kQBytes + (uint32_t)x.nrows * kHeads * 4u);
#pragma unroll
          for (int pp = 0; pp < P; ++pp)    // one box of G rows' heads per pass
            tma_load_2d(sm.q[qb] + pp * G * kQBytes, &tm_q, 0, (x.r0 + pp * G) * kHeads,
                        &sm.qfull[qb]);
          bulk_g2s(sm.w[qb], w + (int64_t)x.r0 * kHeads, (uint32_t)x.nrows * kHeads * 4u,
                   &sm.qfull[qb]);
          ++icount;
          for (int k = 0; k < x.ntiles; ++k, ++gt) {
            const int stg = gt % kStages;
            if (gt >= kStages &&
                !mbar_wait(&sm.empty[stg], (uint32_t)((gt / kStages) - 1) & 1u)) {
              raise_flag(flags, DSA_FLAG_TIMEOUT);
              sm.abort = 1;
              break;
            }
            if (aborted(sm)) break;
            mbar_expect_tx(&sm.full[stg], kTileBytes);
            const uint32_t tok0 = tok_lo + (uint32_t)k * kTile;
            for (int j = 0; j < boxes; ++j) {
              const uint32_t l0 = tok0 + (uint32_t)(j * box_rows);   // first slot of the box
              uint32_t off;
              const int blk = (int)fdivmod(l0, fbs, &off);
              int y = oob_y;
              if (blk < blk_end) {          // a block holding slots of the range
                const int64_t p = sm.pblk[blk - blk0];
                if (p >= 0 && p * block_size + off + box_rows <= n_slots)
                  y = (int)((int64_t)x.s * n_slots + p * block_size + off);
                else
                  bad = true;
              }
              tma_load_2d(sm.k[stg] + (uint32_t)j * box_rows * kDim, &tm_k, 0, y, &sm.full[stg]);
            }
          }
        }
      }
    }
    // Drain: every issued copy has landed before the CTA can exit.
    if (lane == 0) {
      for (int i = max(0, icount - 2); i < icount; ++i)
        mbar_wait(&sm.qfull[i & 1], (uint32_t)(i >> 1) & 1u);
      for (int k = max(0, gt - kStages); k < gt; ++k)
        mbar_wait(&sm.full[k % kStages], (uint32_t)(k / kStages) & 1u);
    }
  } else if (warp == Cfg::kMma) {
    // ---- MMA issuer -------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f8(G * kHeads);
      bool ok = true;
      int gt = 0, icount = 0;
      for (int it = blockIdx.x; ok && it < nitems && !aborted(sm); it += gridDim.x) {
        const Item<R> x = make_item<R>(it, rows, groups, chunks, row_starts, row_ends, ld, sh, &bad);
        if (x.ntiles == 0) continue;
        const int qb = icount & 1;
        if (!mbar_wait(&sm.qfull[qb], (uint32_t)(icount >> 1) & 1u)) { ok = false; break; }
        ++icount;
#ifdef DSA_TEST_STALLED_COPY
        // The test-only build (never libdsa.so): before its first MMA the
        // thread waits on an mbarrier armed for 16 bytes that no copy delivers;
        // every real copy still lands on its own barrier, this wait runs out.
        if (icount == 1) {
          mbar_expect_tx(&sm.stall, 16u);
          if (!mbar_wait(&sm.stall, 0)) { ok = false; break; }
        }
#endif
        for (int kt = 0; kt < x.ntiles; ++kt, ++gt) {
          constexpr int NB = Cfg::kAccBufs;
          const int stg = gt % kStages;
          if (!mbar_wait(&sm.full[stg], (uint32_t)(gt / kStages) & 1u)) { ok = false; break; }
          const uint64_t kdesc = sw128_desc(sm.k[stg]);
#pragma unroll 1
          for (int pp = 0; pp < P; ++pp) {   // one accumulator per pass
            const int u = gt * P + pp, b = u % NB;
            if (u >= NB && !mbar_wait(&sm.accempty[b], (uint32_t)((u / NB) - 1) & 1u)) { ok = false; break; }
            if (aborted(sm)) { ok = false; break; }
            tc_fence_after();
            const uint64_t qdesc = sw128_desc(sm.q[qb] + pp * G * kQBytes);
#pragma unroll
            for (int kk = 0; kk < kDim / 32; ++kk)   // 32 fp8 = 32 bytes = 2 descriptor units
              mma_f8(tmem + (uint32_t)b * Cfg::kAccCols, kdesc + 2u * kk, qdesc + 2u * kk, idesc,
                     kk > 0);
            mma_commit(&sm.accfull[b]);
          }
          if (!ok) break;
          mma_commit(&sm.empty[stg]);        // after every pass over the tile
        }
        mma_commit(&sm.qfree[qb]);   // the item's query slot, once its MMAs are done
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
    // ---- epilogue: warp e reads lanes 32 (e % 4) .. + 31 for row e / 4 -----
    const int quarter = warp & 3, g = warp >> 2;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int gt = 0, icount = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < nitems && !aborted(sm); it += gridDim.x) {
      const Item<R> x = make_item<R>(it, rows, groups, chunks, row_starts, row_ends, ld, sh, &bad);
      if (x.ntiles == 0) continue;
      const int qb = icount & 1;
      if (!mbar_wait(&sm.qfull[qb], (uint32_t)(icount >> 1) & 1u)) { ok = false; break; }
      ++icount;
      // This warp's row of each pass and its range (selected with constant
      // indices, so that the item stays in registers); empty past the batch.
      int64_t my_lo[P], my_hi[P];
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        my_lo[pp] = my_hi[pp] = 0;
#pragma unroll
        for (int gg = 0; gg < R; ++gg)
          if (gg == pp * G + g && gg < x.nrows) {
            my_lo[pp] = x.lo[gg];
            my_hi[pp] = x.hi[gg];
          }
      }
      for (int kt = 0; kt < x.ntiles; ++kt, ++gt) {
        const int64_t l = (x.t_lo + kt) * kTile + quarter * 32 + lane;
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
          constexpr int NB = Cfg::kAccBufs;
          const int u = gt * P + pp, b = u % NB;
          if (!mbar_wait(&sm.accfull[b], (uint32_t)(u / NB) & 1u)) { ok = false; break; }
          if (aborted(sm)) { ok = false; break; }
          tc_fence_after();
          const int row = pp * G + g;      // row of the item
          // Four partial sums (heads h mod 4) as two packed pairs, so the
          // dependent chain is 16 deep; the 64 head sums are read 32 at a time.
          float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int hh = 0; hh < kHeads; hh += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + (uint32_t)b * Cfg::kAccCols + (uint32_t)(g * kHeads + hh),
                      v);
            const float4* wv = reinterpret_cast<const float4*>(sm.w[qb] + row * kHeads + hh);
#pragma unroll
            for (int h4 = 0; h4 < 8; ++h4) {
              const float4 ww = wv[h4];
              a01 = ffma2(make_float2(ww.x, ww.y),
                          make_float2(fmaxf(__uint_as_float(v[4 * h4 + 0]), 0.f),
                                      fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f)),
                          a01);
              a23 = ffma2(make_float2(ww.z, ww.w),
                          make_float2(fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f),
                                      fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f)),
                          a23);
            }
          }
          const float acc = (a01.x + a01.y) + (a23.x + a23.y);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive1(&sm.accempty[b]);
          if (l >= my_lo[pp] && l < my_hi[pp])
            logits[((int64_t)x.s * rows + x.r0 + row) * ld + l] = acc;
        }
        if (!ok) break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&sm.qfree[qb]);   // done with the item's weights
    }
    if (!ok) {
      if (lane == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
      sm.abort = 1;
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);
  tc_fence_before();
  __syncthreads();
  if (warp == Cfg::kProducer) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(Cfg::kTmemCols)
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
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(weights) ||
      (reinterpret_cast<uintptr_t>(logits) & 3u))
    return DSA_ERR_INVALID_ARG;
  const int box_rows = block_size < 64 ? block_size : 64;
  // Four rows per MMA when every row must read the same request's keys.
  const bool grouped = reqs == 1 && rows >= 4;
  CUtensorMap tm_k, tm_q;
  if (!encode_rows(&tm_k, k_cache, (uint64_t)S * (uint64_t)n_slots, (uint32_t)box_rows) ||
      !encode_rows(&tm_q, q, (uint64_t)rows * kHeads, (uint32_t)(grouped ? 4 : 1) * kHeads))
    return DSA_ERR_CUDA;
  const int chunks =
      (int)((ld + (int64_t)kTile * kTilesPerItem - 1) / ((int64_t)kTile * kTilesPerItem));
  const int R = grouped ? 8 : 1;   // rows per item: G rows per MMA times P passes
  const int64_t nitems = (int64_t)S * ((rows + R - 1) / R) * chunks;
  if (nitems > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  auto launch = [&](auto kern, int threads, int per_sm, size_t smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return DSA_ERR_CUDA;
    // Ungrouped items (one row each, uneven lengths) go one per CTA, so the
    // hardware's block scheduler balances them; grouped ones share one
    // persistent CTA per SM.
    const int grid = per_sm > 1 ? (int)nitems : (int)std::min<int64_t>(nitems, (int64_t)sms * per_sm);
    const cudaError_t e = launch_kernel(kern, dim3((unsigned)grid), dim3(threads), smem, stream, 0,
                                        tm_k, tm_q, weights, block_table, reqs, max_blocks,
                                        block_size, box_rows, n_slots, row_to_req, row_starts,
                                        row_ends, rows, S, ld, chunks, (int)nitems, logits,
                                        err_flags, ShardMath(S, I), FastDiv((uint32_t)block_size));
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  };
  if (grouped)
    return launch(indexer_logits_kernel<4, 2>, LogitsCfg<4, 2>::kThreads, 1,
                  sizeof(LogitsSmem<4, 2>) + 1024);
  return launch(indexer_logits_kernel<1, 1>, LogitsCfg<1, 1>::kThreads, 2,
                sizeof(LogitsSmem<1, 1>) + 1024);
}
