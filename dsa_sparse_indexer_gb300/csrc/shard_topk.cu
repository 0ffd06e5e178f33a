// Per-shard local top-K of fp32 indexer logits, and candidate packing.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE":
// section 关键源码片段 (`_merge_dcp_topk_global`: the local top-K positions of
// each rank, then (score, global_id) candidates packed as [batch, topk, 2]
// fp32) and section 实现拆解 item 1 (`pack_dcp_topk_candidates_cutedsl`).
//
// One CTA per (shard, row); the winners are written in ascending slot order
// (ties on the score go to the smaller slot, i.e. the smaller global id).
// Local ranges of up to 16384 slots take the throughput kernel below
// (topk_smem_kernel): the range copied into shared memory by TMA, the exact
// threshold from one histogram linear in the score (bins read off the bits
// of one FFMA) and a ranking of its threshold bin (fast_select.cuh),
// slot-ordered placement through shared memory.
// Longer ranges are staged in shared memory with bulk async copies (TMA) or
// read from global memory, and a radix select with an ordered ballot sweep
// picks the winners (shard_topk_kernel, local_topk.cuh).  The standalone pack
// gathers candidates for given local indices.
#include "checks.h"
#include "common.cuh"
#include "fast_select.cuh"
#include "local_topk.cuh"
#include "reg_topk.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kVec = 8;   // register path: local ranges up to 16384 elements
using RT = RegTopk<kTopkThreads, kVec>;

struct TopkSmem {
  LocalTopkSmem loc;
  RegEmitSmem<kTopkThreads, kVec> es;
  uint32_t list[kListCap];   // keys of the threshold bin
};

__host__ __device__ constexpr size_t topk_stage_offset() {
  return (sizeof(TopkSmem) + 127) & ~size_t(127);
}

__device__ __forceinline__ void write_pad(int32_t* out_idx, float2* out_cand, int j) {
  if (out_idx) out_idx[j] = -1;
  if (out_cand) out_cand[j] = make_float2(-INFINITY, __int_as_float(-1));
}

template <bool kPack>
__global__ void __launch_bounds__(kTopkThreads, 2)
    shard_topk_kernel(const float* __restrict__ logits, int64_t ld, int rows, int S, int I,
                      int K, const int32_t* __restrict__ row_starts,
                      const int32_t* __restrict__ row_ends, int32_t* __restrict__ local_idx,
                      float* __restrict__ cand, uint32_t* flags, int stage_cap,
                      const ShardMath sh) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(smem_raw);
  float* stage = reinterpret_cast<float*>(smem_raw + topk_stage_offset());

  const int tid = threadIdx.x;
  const int s = blockIdx.x / rows, r = blockIdx.x - s * rows;
  const float* row = logits + ((int64_t)s * rows + r) * ld;

  // Global range -> this shard's local range.
  int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  int64_t lo = sh.local_len((uint32_t)st, s), hi = sh.local_len((uint32_t)en, s);
  if (hi > ld) { hi = ld; bad = true; }
  if (lo > hi) { lo = hi; bad = true; }
  if (bad && tid == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
  const int n = (int)(hi - lo);

  int32_t* out_idx = local_idx ? local_idx + ((int64_t)s * rows + r) * K : nullptr;
  float2* out_cand = kPack ? reinterpret_cast<float2*>(cand) + ((int64_t)r * S + s) * K : nullptr;

  if (n <= K) {  // every slot is selected: slots lo..hi-1 in order, then padding
    for (int j = tid; j < K; j += kTopkThreads) {
      if (j < n) {
        const int64_t l = lo + j;
        if (out_idx) out_idx[j] = (int32_t)l;
        if (kPack) out_cand[j] = make_float2(row[l], __int_as_float((int)sh.global_id(s, (uint32_t)l)));
      } else {
        write_pad(out_idx, out_cand, j);
      }
    }
    return;
  }

  const int64_t base = lo & ~int64_t(3);
  if (hi - base <= RT::kCap) {
    uint32_t key[kVec][4];
    load_keys<kTopkThreads, kVec>(row, lo, hi, key);
    int eq;
    const SelectResult res = select_regs<kTopkThreads, kVec>(key, K, sm.loc.sel, sm.list, sm.es,
                                                             &eq);
    emit_winners<kTopkThreads, kVec>(key, res.thr, res.take_eq, sm.es,
                                     [&](int p, int e, uint32_t) {
      if (p >= K) return;
      const uint32_t l = (uint32_t)(base + e);
      if (out_idx) out_idx[p] = (int32_t)l;
      if (kPack) out_cand[p] = make_float2(row[l], __int_as_float((int)sh.global_id(s, l)));
    });
    return;
  }
  bool ok;
  const float* data = stage_local_range(row, lo, hi, stage, stage_cap, sm.loc, flags, &ok);
  if (!ok) return;
  local_topk_emit<kTopkThreads>(data, n, K, sm.loc, [&](int p, int i, float v) {
    const uint32_t l = (uint32_t)(lo + i);
    if (out_idx) out_idx[p] = (int32_t)l;
    if (kPack) out_cand[p] = make_float2(v, __int_as_float((int)sh.global_id(s, l)));
  });
}

// ---------------------------------------------------------------------------
// Throughput path for local ranges of up to 4 V NT slots (NT = 256 threads
// with V = 8 float4 rows each up to 8192 slots, five CTAs per SM; 512 up to
// 16384, two CTAs per SM).  One bulk copy (TMA) brings the row's range into
// shared memory, completing on an mbarrier; thread tid owns float4 rows
// j NT + tid (slot e = base + 4 (j NT + tid) + c) and reads them from shared
// memory in every pass, the first of which writes -inf over its slots outside
// [lo, hi).  No score is held in registers between passes, which leaves room
// for five CTAs of 256 threads an SM.  The exact threshold (score, slot)
// comes from fast_select (fast_select.cuh: a histogram of the scores linear
// in the score over their range, a ranking of the threshold bin): a slot
// wins if its score is above the threshold score, or equal to it at a slot
// no later than the threshold slot (scores compare as floats: -0.0 ties
// +0.0, as their keys do, and each keeps its own sign in the candidate).
// The winners are then placed in slot order: per-thread counts for each of
// the V float4 rows, packed four to a word, take one warp scan a word, and a
// small table gives each (row, warp) its output offset; each thread drops
// its winners' slots at their output positions in shared memory, and all
// threads then write the outputs with coalesced stores, the scores read back
// from the copy.  Rows with an infinite score or a crowded threshold bin
// rank the copy with the radix select (local_topk.cuh).
// ---------------------------------------------------------------------------
constexpr int kTMaxK = 2048;     // largest K

// Writes winner p of a (shard, row): local slot l and the packed candidate.
template <bool kPack>
struct TopkEmitter {
  const float* row;
  int32_t* out_idx;
  float2* out_cand;
  int K, s;
  ShardMath sh;
  __device__ __forceinline__ void operator()(int p, uint32_t l, float v) const {
    if (p >= K) return;
    if (out_idx) out_idx[p] = (int32_t)l;
    if (kPack) out_cand[p] = make_float2(v, __int_as_float((int)sh.global_id(s, l)));
  }
};

template <int NT, int V>
struct TopkSmemLayout {
  float4 sc[V * NT];               // slots [base, base + 4 V NT) of the row
  union {
    struct {
      // The selection's bins are dead once the threshold is known: the
      // winners' slots are staged by output position in their place.
      FastSelectSmem sel;
      uint32_t wt[V / 4][NT / 32]; // packed per-row winner counts of each warp
      int off[V][NT / 32];         // output offset of each (float4 row, warp)
    } f;
    LocalTopkSmem loc;             // fallback: radix select over the copy
  };
  uint64_t bar;
#ifdef DSA_TEST_STALLED_COPY
  uint64_t stall;                  // test build: armed for bytes no copy delivers
#endif
};

static_assert(kFsBins >= kTMaxK, "the staged winners fit the bins");
static_assert(sizeof(TopkSmemLayout<256, 8>) <= 44 * 1024, "five CTAs of 256 threads an SM");
static_assert(sizeof(TopkSmemLayout<512, 8>) <= 113 * 1024, "two CTAs of 512 threads an SM");

// CTAs an SM: five of 256 threads (44 KB of shared memory each), two of 512.
template <int NT>
constexpr int topk_smem_min_blocks() { return NT == 256 ? 5 : 1024 / NT; }

template <int NT, int V, bool kPack>
__global__ void __launch_bounds__(NT, topk_smem_min_blocks<NT>())
    topk_smem_kernel(const float* __restrict__ logits, int64_t ld, int rows, int S, int I, int K,
                     const int32_t* __restrict__ row_starts, const int32_t* __restrict__ row_ends,
                     int32_t* __restrict__ local_idx, float* __restrict__ cand, uint32_t* flags,
                     const ShardMath sh) {
  static_assert(V % 4 == 0 && V <= 8, "per-row winner counts are packed four to a word");
  constexpr int NW = V / 4;
  constexpr int W = NT / 32;
  extern __shared__ __align__(16) unsigned char topk_smem_raw[];
  TopkSmemLayout<NT, V>& sm = *reinterpret_cast<TopkSmemLayout<NT, V>*>(topk_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.x, s = blockIdx.y;
  const float* row = logits + ((int64_t)s * rows + r) * ld;

  // Global range -> this shard's local range (ld <= INT32_MAX: slots fit int).
  int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  int64_t lo64 = sh.local_len((uint32_t)st, s), hi64 = sh.local_len((uint32_t)en, s);
  if (hi64 > ld) { hi64 = ld; bad = true; }
  if (lo64 > hi64) { lo64 = hi64; bad = true; }
  if (bad && tid == 0) raise_flag(flags, DSA_FLAG_BOUNDS);
  const int lo = (int)lo64, hi = (int)hi64, n = hi - lo;

  auto make_emit = [&]() {
    return TopkEmitter<kPack>{
        row, local_idx ? local_idx + ((int64_t)s * rows + r) * K : nullptr,
        kPack ? reinterpret_cast<float2*>(cand) + ((int64_t)r * S + s) * K : nullptr, K, s, sh};
  };
  if (n <= K) {  // every slot is selected: slots lo..hi-1 in order, then padding
    const TopkEmitter<kPack> emit = make_emit();
    for (int j = tid; j < K; j += NT) {
      if (j < n) emit(j, (uint32_t)(lo + j), __ldg(row + lo + j));
      else write_pad(emit.out_idx, emit.out_cand, j);
    }
    return;
  }
  // The copy: [base, hi rounded up to 4) (inside the row: ld % 4 == 0; at
  // most 4 V NT slots, which the launch guarantees with ld <= 4 V NT).
  const int base = lo & ~3, top = (hi + 3) & ~3;
  const uint32_t bytes = (uint32_t)(top - base) * 4u;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
#ifdef DSA_TEST_STALLED_COPY
    mbar_init(&sm.stall, 1);
#endif
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {   // in pieces of at most 16 KB, all completing on one barrier
    mbar_expect_tx(&sm.bar, bytes);
    for (uint32_t off = 0; off < bytes; off += 16384u)
      bulk_g2s(reinterpret_cast<unsigned char*>(sm.sc) + off,
               reinterpret_cast<const unsigned char*>(row + base) + off, min(16384u, bytes - off),
               &sm.bar);
  }
#ifdef DSA_TEST_STALLED_COPY
  if (tid == 0) mbar_expect_tx(&sm.stall, 16u);
#endif
  bool good = mbar_wait(&sm.bar, 0);
#ifdef DSA_TEST_STALLED_COPY
  good &= mbar_wait(&sm.stall, 0);
#endif
  if (__syncthreads_or(!good)) {
    if (tid == 0) raise_flag(flags, DSA_FLAG_TIMEOUT);
    mbar_wait(&sm.bar, 0);   // the copy must land before the CTA's memory goes
    return;
  }

  // Range pass: each thread's float4 rows, -inf written over its slots
  // outside [lo, hi) (it is the only reader of them until the next barrier);
  // the rows stay in registers for the histogram, the next pass.
  float fmn = INFINITY, fmx = -INFINITY;
  float4 rv[V];
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int q = j * NT + tid, e0 = base + 4 * q;
    if (e0 >= lo && e0 + 4 <= hi) {
      rv[j] = sm.sc[q];
      fmn = fminf(fminf(fminf(fminf(fmn, rv[j].x), rv[j].y), rv[j].z), rv[j].w);
      fmx = fmaxf(fmaxf(fmaxf(fmaxf(fmx, rv[j].x), rv[j].y), rv[j].z), rv[j].w);
    } else {
      float4 v = e0 < top ? sm.sc[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      float* e = reinterpret_cast<float*>(&v);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const bool in = e0 + c >= lo && e0 + c < hi;
        e[c] = in ? e[c] : -INFINITY;
        fmn = in ? fminf(fmn, e[c]) : fmn;
        fmx = in ? fmaxf(fmx, e[c]) : fmx;
      }
      sm.sc[q] = v;
      rv[j] = v;
    }
  }
  const float* scf = reinterpret_cast<const float*>(sm.sc);
  auto slot = [&](int j, int c) { return (uint32_t)(base + (j * NT + tid) * 4 + c); };
  auto get4 = [&](int j) { return sm.sc[j * NT + tid]; };
  auto score_at = [&](uint32_t l) { return scf[l - (uint32_t)base]; };

  FastSelectResult fs;
  auto get4h = [&](int j) { return rv[j]; };
  if (!fast_select<NT, V>(get4h, get4, K, fmn, fmx, slot, score_at, sm.f.sel, &fs)) {
    __syncthreads();   // the fallback's shared memory overlaps the selection's
    const TopkEmitter<kPack> emit = make_emit();
    local_topk_emit<NT>(scf + (lo - base), n, K, sm.loc,
                        [&](int p, int i, float v) { emit(p, (uint32_t)(lo + i), v); });
    return;
  }

  const float thr = fs.thr;
  const uint32_t last = fs.last;
  uint32_t wmask = 0u;   // bit 4 j + c: slot (j, c) wins
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float4 v = get4(j);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float x = f4at(v, c);
      wmask |= (uint32_t)(fs.eq == 1 ? x >= thr : (x > thr || (x == thr && slot(j, c) <= last)))
               << (4 * j + c);
    }
  }
  uint32_t pk[NW], inc[NW];   // winners per float4 row j: word j / 4, 8 bits each
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    pk[w] = 0u;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      pk[w] |= (uint32_t)__popc((wmask >> (4 * (4 * w + jj))) & 0xfu) << (8 * jj);
    inc[w] = pk[w];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t y = __shfl_up_sync(kFull, inc[w], o);
      if (lane >= o) inc[w] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int w = 0; w < NW; ++w) sm.f.wt[w][warp] = inc[w];
  }
  __syncthreads();
  if (warp == 0) {
    int row_base = 0;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t wt = lane < W ? sm.f.wt[j / 4][lane] : 0u;
      const int c = (int)((wt >> (8 * (j % 4))) & 0xffu);
      const int incl = warp_inclusive_scan(c);
      if (lane < W) sm.f.off[j][lane] = row_base + incl - c;
      row_base += __shfl_sync(kFull, incl, 31);
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < V; ++j) {
    int p = sm.f.off[j][warp] + (int)(((inc[j / 4] - pk[j / 4]) >> (8 * (j % 4))) & 0xffu);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (wmask >> (4 * j + c) & 1u) {
        if (p < K) sm.f.sel.bins[p] = slot(j, c);
        ++p;
      }
  }
  __syncthreads();
  const TopkEmitter<kPack> emit = make_emit();
  for (int p = tid; p < K; p += NT) {
    const uint32_t l = sm.f.sel.bins[p];
    emit(p, l, scf[l - (uint32_t)base]);
  }
}

// Standalone pack: cand[r][s*K + j] from local_idx[s][r][j].  Each thread
// handles four consecutive j (K % 4 == 0): one 16-byte index load, four
// gathers from the logits, two 16-byte candidate stores.
__global__ void __launch_bounds__(256)
    pack_kernel(const float* __restrict__ logits, int64_t ld,
                const int32_t* __restrict__ local_idx, int rows, int S, int K,
                float* __restrict__ cand, uint32_t* flags, const ShardMath sh) {
  const int64_t quads = (int64_t)S * rows * K / 4;
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= quads) return;
  const int64_t flat = q * 4;                 // index into [S][rows][K]
  const int j = (int)(flat % K);
  const int64_t sr = flat / K;
  const int r = (int)(sr % rows), s = (int)(sr / rows);
  const int4 li = *reinterpret_cast<const int4*>(local_idx + flat);
  const float* row = logits + ((int64_t)s * rows + r) * ld;
  const int l4[4] = {li.x, li.y, li.z, li.w};
  float2 o[4];
  bool bad = false;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int l = l4[u];
    if (l >= 0 && l < ld) {
      o[u] = make_float2(__ldg(row + l), __int_as_float((int)sh.global_id(s, (uint32_t)l)));
    } else {
      bad |= l >= ld;
      o[u] = make_float2(-INFINITY, __int_as_float(-1));
    }
  }
  if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);
  float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float2*>(cand) + ((int64_t)r * S + s) * K + j);
  dst[0] = make_float4(o[0].x, o[0].y, o[1].x, o[1].y);
  dst[1] = make_float4(o[2].x, o[2].y, o[3].x, o[3].y);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Scalar checks first; with rows == 0 nothing is read, so pointers may be NULL.
dsa_status check_common(const float* logits, int64_t ld, int rows, int S, int I, int K) {
  if (rows < 0 || ld < 4 || (ld & 3)) return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > DSA_MAX_SHARDS || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (ld > (int64_t)INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)rows * S > (int64_t)INT32_MAX || (int64_t)I * S > (int64_t)INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (rows > 0 && (!logits || !aligned16(logits))) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

template <bool kPack>
dsa_status launch_topk(const float* logits, int64_t ld, int rows, int S, int I, int K,
                       const int32_t* row_starts, const int32_t* row_ends, int32_t* local_idx,
                       float* cand, uint32_t* err_flags, cudaStream_t stream) {
  const ShardMath shm(S, I);
  if (ld <= 32 * 512) {
    auto launch_fast = [&](auto kern, int nt) {
      const cudaError_t e = launch_kernel(kern, dim3((unsigned)rows, (unsigned)S), dim3((unsigned)nt), 0,
                                          stream, 0, logits, ld, rows, S, I, K, row_starts,
                                          row_ends, local_idx, cand, err_flags, shm);
      return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
    };
    auto launch_smem = [&](auto kern, int nt, size_t smem) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
        return DSA_ERR_CUDA;
      const cudaError_t e = launch_kernel(kern, dim3((unsigned)rows, (unsigned)S),
                                          dim3((unsigned)nt), smem, stream, 0, logits, ld, rows,
                                          S, I, K, row_starts, row_ends, local_idx, cand,
                                          err_flags, shm);
      return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
    };
    if (ld <= 32 * 256)
      return launch_smem(topk_smem_kernel<256, 8, kPack>, 256, sizeof(TopkSmemLayout<256, 8>));
    return launch_smem(topk_smem_kernel<512, 8, kPack>, 512, sizeof(TopkSmemLayout<512, 8>));
  }
  // Rows that fit the register path need no staging area.
  const int stage_cap = ld <= RT::kCap ? 0 : (ld < kStageCapElems ? (int)ld : kStageCapElems);
  const size_t smem = topk_stage_offset() + (size_t)stage_cap * sizeof(float);
  auto kern = shard_topk_kernel<kPack>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  const cudaError_t e = launch_kernel(kern, dim3((unsigned)(rows * S)), dim3(kTopkThreads), smem,
                                      stream, 0, logits, ld, rows, S, I, K, row_starts, row_ends,
                                      local_idx, cand, err_flags, stage_cap, ShardMath(S, I));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_shard_topk(const float* logits, int64_t ld, int rows, int S, int I,
                                     int K, const int32_t* row_starts, const int32_t* row_ends,
                                     int32_t* local_idx, uint32_t* err_flags,
                                     cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (rows == 0) return DSA_OK;
  if (!row_ends || !local_idx) return DSA_ERR_INVALID_ARG;
  return launch_topk<false>(logits, ld, rows, S, I, K, row_starts, row_ends, local_idx, nullptr,
                            err_flags, stream);
}

dsa_status dsa::check_shard_topk_pack(const float* logits, int64_t ld, int rows, int S, int I,
                                      int K, const int32_t* row_ends, const float* cand) {
  const dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK || rows == 0) return st;
  if (!row_ends || !cand || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

extern "C" dsa_status dsa_shard_topk_pack(const float* logits, int64_t ld, int rows, int S,
                                          int I, int K, const int32_t* row_starts,
                                          const int32_t* row_ends, int32_t* local_idx,
                                          float* cand, uint32_t* err_flags,
                                          cudaStream_t stream) {
  const dsa_status st = check_shard_topk_pack(logits, ld, rows, S, I, K, row_ends, cand);
  if (st != DSA_OK || rows == 0) return st;
  return launch_topk<true>(logits, ld, rows, S, I, K, row_starts, row_ends, local_idx, cand,
                           err_flags, stream);
}

extern "C" dsa_status dsa_pack_candidates(const float* logits, int64_t ld,
                                          const int32_t* local_idx, int rows, int S, int I,
                                          int K, float* cand, uint32_t* err_flags,
                                          cudaStream_t stream) {
  dsa_status st = check_common(logits, ld, rows, S, I, K);
  if (st != DSA_OK) return st;
  if (rows == 0) return DSA_OK;
  if (!local_idx || !cand || !aligned16(local_idx) || !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  const int64_t quads = (int64_t)S * rows * K / 4;
  const int64_t blocks = (quads + 255) / 256;
  if (blocks > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  const cudaError_t e = launch_kernel(pack_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 0,
                                      logits, ld, local_idx, rows, S, K, cand, err_flags,
                                      ShardMath(S, I));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
