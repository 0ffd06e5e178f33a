// The indexer path for one row per thread-block cluster: local top-K of every
// shard, candidate exchange, stable merge and slot conversion in one kernel.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 关键源码片段 (`_merge_dcp_topk_global`: local top-K on every rank,
// (score, global_id) candidates, all_gather, stable selector) and section
// 实现拆解 items 1, 2 and 4 (pack, merge, convert with compaction).
//
// The cluster holds S CTAs, CTA rank s playing DCP rank s.  Each CTA stages its
// shard's local range in shared memory (bulk async copies) and selects its K
// local candidates as in the per-shard kernel, keeping them in shared memory as
// 64-bit rank keys (score_key << 32 | ~global_id).  The pages' all_gather of
// candidates becomes reads of the other CTAs' shared memory (DSMEM): the
// cluster runs a radix select over all S*K candidates with per-CTA histograms
// summed across the cluster, each CTA sorts the global winners it holds (a
// bitonic sort in shared memory), and a winner's global rank is its rank among
// its own CTA's winners plus, for every other CTA, the number of that CTA's
// winners ranked above it (binary search in a local copy of their sorted
// lists).  A shard's winners in rank order are exactly its compacted slots, so
// each CTA maps them through its own block table and writes them directly.
#include <cooperative_groups.h>

#include "common.cuh"
#include "local_topk.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kFusedThreads = 512;
constexpr int kMaxK = 2048;
constexpr int kMaxCluster = 8;

struct FusedSmem {
  LocalTopkSmem loc;
  uint32_t chist[2048];             // this CTA's share of a cluster-wide histogram
  unsigned long long cand[kMaxK];   // local candidates as rank keys, slot order
  int scan[64];
  int wr[kMaxCluster], off[kMaxCluster];
  int m, w, total, tied, nwin, bin, above, count;
};

__host__ __device__ constexpr size_t fused_dyn_offset() {
  return (sizeof(FusedSmem) + 127) & ~size_t(127);
}

__device__ __forceinline__ unsigned long long rank_key(float v, int gid) {
  return ((unsigned long long)score_key(v) << 32) | (unsigned long long)(~(uint32_t)gid);
}

// Cluster-wide version of radix_select (select.cuh): the need-th largest key
// among all CTAs' elements i in [0, m) with key_at(i, &k) true; every CTA of
// the cluster computes the same result.  Two cluster barriers per digit.
template <typename KeyAt>
__device__ SelectResult cluster_select(cg::cluster_group& cluster, int nranks, int m, int need,
                                       KeyAt key_at, FusedSmem& sm) {
  constexpr int NT = kFusedThreads;
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    const int per = nb / NT;
    for (int b = tid; b < nb; b += NT) sm.chist[b] = 0u;
    __syncthreads();
    for (int i = tid; i < m; i += NT) {
      uint32_t k;
      if (key_at(i, k) && (k & mask) == prefix) atomicAdd(&sm.chist[(k >> shift) & (nb - 1)], 1u);
    }
    cluster.sync();
    int c[4] = {0, 0, 0, 0};
    for (int rk = 0; rk < nranks; ++rk) {
      const uint32_t* h = cluster.map_shared_rank(sm.chist, rk);
      for (int j = 0; j < per; ++j) c[j] += (int)h[nb - 1 - (tid * per + j)];
    }
    int local = 0;
    for (int j = 0; j < per; ++j) local += c[j];
    int total;
    int running = block_exclusive_scan(local, sm.scan, &total);
    for (int j = 0; j < per; ++j) {
      if (running < need && running + c[j] >= need) {
        sm.bin = nb - 1 - (tid * per + j);
        sm.above = running;
        sm.count = c[j];
      }
      running += c[j];
    }
    __syncthreads();
    const int b = sm.bin, above = sm.above, count = sm.count;
    need -= above;
    prefix |= (uint32_t)b << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    cluster.sync();  // every CTA is done reading chist before it is cleared again
    if (count == need) return SelectResult{prefix - 1u, 0};
  }
  return SelectResult{prefix, need};
}

// Entries of a descending list that rank above `key` (all keys distinct).
__device__ __forceinline__ int count_above(const unsigned long long* list, int len,
                                           unsigned long long key) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (list[mid] > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kFusedThreads, 2)
    fused_kernel(const float* __restrict__ logits, int64_t ld, int rows, int S, int I, int K,
                 const int32_t* __restrict__ row_starts, const int32_t* __restrict__ row_ends,
                 const int32_t* __restrict__ bt, int reqs, int max_blocks, int bs,
                 const int32_t* __restrict__ row_to_req, int32_t* __restrict__ ids,
                 float* __restrict__ scores, int32_t* __restrict__ slots,
                 int32_t* __restrict__ counts, int32_t* __restrict__ local_idx,
                 float* __restrict__ cand_out, uint32_t* flags, int stage_cap) {
  constexpr int NT = kFusedThreads;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(smem_raw);
  unsigned char* dyn = smem_raw + fused_dyn_offset();
  const int tid = threadIdx.x, lane = tid & 31;
  const int s = (int)cluster.block_rank();
  const int r = blockIdx.x / S;
  const float* row = logits + ((int64_t)s * rows + r) * ld;

  // ---- this shard's local range ------------------------------------------
  int64_t st = row_starts ? (int64_t)row_starts[r] : 0, en = row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  int64_t lo = local_len(st, s, S, I), hi = local_len(en, s, S, I);
  if (hi > ld) { hi = ld; bad = true; }
  if (lo > hi) { lo = hi; bad = true; }
  const int n = (int)(hi - lo);
  if (tid == 0) {
    if (bad) raise_flag(flags, DSA_FLAG_BOUNDS);
    sm.m = min(n, K);
    sm.tied = 0;
    sm.nwin = 0;
  }
  int32_t* out_idx = local_idx ? local_idx + ((int64_t)s * rows + r) * K : nullptr;
  float2* out_cand = cand_out ? reinterpret_cast<float2*>(cand_out) + ((int64_t)r * S + s) * K
                              : nullptr;
  __syncthreads();

  // ---- a1 + a2: local top-K, kept as rank keys -----------------------------
  if (n <= K) {
    for (int j = tid; j < K; j += NT) {
      if (j < n) {
        const int64_t l = lo + j;
        const float v = row[l];
        const int gid = (int)global_of(s, l, S, I);
        sm.cand[j] = rank_key(v, gid);
        if (out_idx) out_idx[j] = (int32_t)l;
        if (out_cand) out_cand[j] = make_float2(v, __int_as_float(gid));
      } else {
        if (out_idx) out_idx[j] = -1;
        if (out_cand) out_cand[j] = make_float2(-INFINITY, __int_as_float(-1));
      }
    }
  } else {
    bool ok;
    const float* data = stage_local_range(row, lo, hi, reinterpret_cast<float*>(dyn), stage_cap,
                                          sm.loc, flags, &ok);
    local_topk_emit<NT>(data, n, K, sm.loc, [&](int p, int i, float v) {
      const int64_t l = lo + i;
      const int gid = (int)global_of(s, l, S, I);
      sm.cand[p] = rank_key(v, gid);
      if (out_idx) out_idx[p] = (int32_t)l;
      if (out_cand) out_cand[p] = make_float2(v, __int_as_float(gid));
    });
  }
  cluster.sync();  // every CTA's candidates are in place

  // ---- a3: select the global winners across the cluster --------------------
  if (tid == 0) {
    int t = 0;
    for (int rk = 0; rk < S; ++rk) t += *cluster.map_shared_rank(&sm.m, rk);
    sm.total = t;
  }
  __syncthreads();
  const int total = sm.total, m = sm.m;
  const bool all = total <= K;
  bool tie = false;
  uint32_t thr1 = 0, thr2 = 0;
  if (!all) {
    auto key1 = [&](int i, uint32_t& k) {
      k = (uint32_t)(sm.cand[i] >> 32);
      return true;
    };
    const SelectResult a = cluster_select(cluster, S, m, K, key1, sm);
    thr1 = a.thr;
    if (a.take_eq > 0) {
      int e = 0;
      for (int i = tid; i < m; i += NT) e += (uint32_t)(sm.cand[i] >> 32) == thr1;
      e = __reduce_add_sync(kFull, e);
      if (lane == 0 && e) atomicAdd(&sm.tied, e);
      cluster.sync();
      int tied = 0;
      for (int rk = 0; rk < S; ++rk) tied += *cluster.map_shared_rank(&sm.tied, rk);
      if (tied > a.take_eq) {
        auto key2 = [&](int i, uint32_t& k) {
          const unsigned long long c = sm.cand[i];
          k = (uint32_t)c;  // ~global id: larger = smaller id
          return (uint32_t)(c >> 32) == thr1;
        };
        const SelectResult b = cluster_select(cluster, S, m, a.take_eq, key2, sm);
        thr2 = b.take_eq > 0 ? b.thr : b.thr + 1u;
        tie = true;
      } else {
        thr1 -= 1u;  // the whole tied group is in
      }
    }
  }

  // This CTA's winners, sorted best first (the staging area is free now).
  unsigned long long* win = reinterpret_cast<unsigned long long*>(dyn);
  unsigned long long* others = win + kMaxK;
  for (int base = 0; base < m; base += NT) {
    const int i = base + tid;
    bool wsel = false;
    unsigned long long key = 0ull;
    if (i < m) {
      key = sm.cand[i];
      const uint32_t k1 = (uint32_t)(key >> 32);
      wsel = all || k1 > thr1 || (tie && k1 == thr1 && (uint32_t)key >= thr2);
    }
    const unsigned msk = __ballot_sync(kFull, wsel);
    int wbase = 0;
    if (lane == 0 && msk) wbase = atomicAdd(&sm.nwin, __popc(msk));
    wbase = __shfl_sync(kFull, wbase, 0);
    const int slot = wbase + __popc(msk & lanemask_lt());
    if (wsel && slot < K) win[slot] = key;
  }
  __syncthreads();
  const int w = min(sm.nwin, K);
  int P = 1;
  while (P < w) P <<= 1;
  for (int j = w + tid; j < P; j += NT) win[j] = 0ull;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int p = tid; p < (P >> 1); p += NT) {
        const int i = 2 * p - (p & (j - 1));
        const int ixj = i + j;
        const bool desc = (i & k) == 0;
        const unsigned long long a = win[i], b = win[ixj];
        if ((a < b) == desc) { win[i] = b; win[ixj] = a; }
      }
      __syncthreads();
    }
  }

  // ---- a4: this shard's winners in rank order are its compacted slots -------
  const int req = row_to_req ? row_to_req[r] : r;
  const bool req_ok = req >= 0 && req < reqs;
  int32_t* dst = slots + ((int64_t)s * rows + r) * K;
  bool slot_bad = false;
  for (int i = tid; i < K; i += NT) {
    int slot = -1;
    if (i < w) {
      const int gid = (int)~(uint32_t)win[i];
      const int64_t l = local_slot_of(gid, S, I);
      const int64_t col = l / bs;
      if (req_ok && col < max_blocks) {
        const int blk = bt[((int64_t)s * reqs + req) * max_blocks + col];
        const int64_t v = (int64_t)blk * bs + l % bs;
        if (blk >= 0 && v <= (int64_t)INT32_MAX) slot = (int)v;
        else slot_bad = true;
      } else {
        slot_bad = true;
      }
    }
    dst[i] = slot;
  }
  if (slot_bad || (!req_ok && w > 0)) raise_flag(flags, DSA_FLAG_BOUNDS);
  if (tid == 0) {
    if (counts) counts[(int64_t)s * rows + r] = w;
    sm.w = w;
  }
  cluster.sync();  // every CTA's sorted winners are published

  // ---- merged ids: rank = own position + winners of other shards above -------
  if (tid < S) sm.wr[tid] = *cluster.map_shared_rank(&sm.w, tid);
  __syncthreads();
  if (tid == 0) {
    int o = 0;
    for (int rk = 0; rk < S; ++rk) {
      sm.off[rk] = o;
      if (rk != s) o += sm.wr[rk];
    }
  }
  __syncthreads();
  for (int rk = 0; rk < S; ++rk) {
    if (rk == s) continue;
    const unsigned long long* remote = cluster.map_shared_rank(win, rk);
    const int len = sm.wr[rk], o = sm.off[rk];
    for (int j = tid; j < len; j += NT)
      if (o + j < kMaxK) others[o + j] = remote[j];
  }
  __syncthreads();
  int32_t* out_ids = ids + (int64_t)r * K;
  float* out_sc = scores ? scores + (int64_t)r * K : nullptr;
  for (int i = tid; i < w; i += NT) {
    const unsigned long long key = win[i];
    int rank = i;
    for (int rk = 0; rk < S; ++rk)
      if (rk != s) rank += count_above(others + sm.off[rk], sm.wr[rk], key);
    if (rank < K) {
      out_ids[rank] = (int32_t)~(uint32_t)key;
      if (out_sc) out_sc[rank] = key_score((uint32_t)(key >> 32));
    }
  }
  if (s == 0) {
    for (int j = min(total, K) + tid; j < K; j += NT) {
      out_ids[j] = -1;
      if (out_sc) out_sc[j] = -INFINITY;
    }
  }
  cluster.sync();  // no CTA leaves while another still reads its shared memory
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status dsa_indexer_fused(const float* logits, int64_t ld, int rows, int S, int I,
                                        int K, const int32_t* row_starts,
                                        const int32_t* row_ends, const int32_t* block_table,
                                        int reqs, int max_blocks, int block_size,
                                        const int32_t* row_to_req, int32_t* ids, float* scores,
                                        int32_t* slots, int32_t* counts, int32_t* local_idx,
                                        float* cand, uint32_t* err_flags, cudaStream_t stream) {
  if (rows < 0 || ld < 4 || (ld & 3) || reqs < 1 || max_blocks < 1 || block_size < 1)
    return DSA_ERR_INVALID_ARG;
  if (S < 1 || S > kMaxCluster || I < 1) return DSA_ERR_UNSUPPORTED;
  if (K != 512 && K != 1024 && K != 2048) return DSA_ERR_UNSUPPORTED;
  if (ld > (int64_t)INT32_MAX || (int64_t)rows * S > (int64_t)INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!logits || !row_ends || !block_table || !ids || !slots || !aligned16(logits))
    return DSA_ERR_INVALID_ARG;
  if (cand && !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  const int stage_cap = ld < kStageCapElems ? (int)ld : kStageCapElems;
  size_t dyn = (size_t)stage_cap * sizeof(float);
  if (dyn < 2 * kMaxK * sizeof(unsigned long long)) dyn = 2 * kMaxK * sizeof(unsigned long long);
  const size_t smem = fused_dyn_offset() + dyn;
  if (cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * S));
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, fused_kernel, logits, ld, rows, S, I, K,
                                           row_starts, row_ends, block_table, reqs, max_blocks,
                                           block_size, row_to_req, ids, scores, slots, counts,
                                           local_idx, cand, err_flags, stage_cap);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
