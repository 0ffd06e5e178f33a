// The indexer path for one row per thread-block cluster: local top-K of every
// shard, candidate exchange, stable merge and slot conversion in one kernel.
//
// PR #46076 report, "[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE",
// section 关键源码片段 (`_merge_dcp_topk_global`: local top-K on every rank,
// (score, global_id) candidates, all_gather, stable selector) and section
// 实现拆解 items 1, 2 and 4 (pack, merge, convert with compaction).
//
// The cluster holds S CTAs, CTA rank s playing DCP rank s.
//  1. Each CTA selects its shard's K local candidates: the local range is held
//     in registers as score keys (reg_topk.cuh; longer ranges are staged in
//     shared memory, local_topk.cuh), and the winners are kept in shared memory
//     as 64-bit rank keys (score_key << 32 | ~global_id).
//  2. The pages' all_gather becomes reads of the other CTAs' shared memory
//     (DSMEM).  A per-binade histogram summed over the cluster sets the floor
//     of 1024 fine bins; each CTA counting-sorts its candidates above the
//     floor into those bins and sorts inside each (small) bin; the fine bins
//     summed over the cluster give the bin b* holding the K-th candidate.
//     Every CTA copies the other CTAs' sorted lists down to b* and resolves
//     the threshold among b*'s few members (the same data, so the same answer
//     everywhere).  Ties on the score go to the smaller global id.
//  3. A shard's winners in rank order are exactly its compacted slots, so
//     each CTA maps them through its own block table and writes them.
//  4. A winner's global rank is its position among its CTA's winners plus,
//     for every other CTA, the number of that CTA's winners ranked above it
//     (binary search in the copied lists); it writes its id at that rank.
//  Rows where a winner-holding bin is crowded (heavy ties) take the exact
//  path instead: a radix select finished over the cluster's gathered
//  threshold bin and a bitonic sort of each CTA's winners.
#include <cooperative_groups.h>
#include <cstddef>

#include "common.cuh"
#include "local_topk.cuh"
#include "reg_topk.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kNT = 512;
constexpr int kVec = 8;                      // 32 keys per thread: local ranges up to 16384
constexpr int kMaxK = 2048;
constexpr int kCandPerThread = kMaxK / kNT;  // 4
constexpr int kMaxCluster = 8;
constexpr int kTableCap = 2048;               // block-table columns kept in shared memory
using RT = RegTopk<kNT, kVec>;
using ull = unsigned long long;

constexpr int kGatherCap = 2 * kMaxK;   // threshold-bin candidates gathered from the cluster
constexpr int kBinCap = 64;             // larger winner-holding bins take the select-and-sort path
constexpr int kNB = 1024;               // fine bins of the one-pass merge
constexpr int kCoarse = 512;            // coarse bins: one per binade of the score (top 9 key bits)
constexpr int kScratch = 3 * kMaxK + kBinCap;   // LB + LS + others, or the heavy-tie gather

struct FusedSmem {
  LocalTopkSmem loc;                 // select scratch (also the staged path's barriers)
  RegEmitSmem<kNT, kVec> es;
  alignas(16) uint32_t chist[2][2048];  // cluster-visible histograms, double-buffered
                                        // (read four bins at a time: 16-byte aligned)
  ull cand[kMaxK];                   // this shard's candidates; later its threshold-bin list
  // Reused in turn: the local select's compacted list (as uint32), the
  // gathered threshold-bin candidates, then win[kMaxK] + others[kMaxK].
  alignas(16) ull scratch[kScratch];
  int32_t sbt[kTableCap];            // this shard's block-table row for the row's request
  int scan[64];
  int wr[kMaxCluster], off[kMaxCluster];
  int m, w, total, tied, nwin, ncl, bin, above, count;
  uint32_t kmin, kmax;             // this CTA's candidate score keys, lowest and highest
  int bstar, bneed, bmax, nown;    // fine-bin merge: threshold bin, rank in it, largest bin
  ull thr64;                       // fine-bin merge: the K-th candidate's rank key
  uint32_t rk_min[kMaxCluster], rk_max[kMaxCluster];
  int rk_m[kMaxCluster], moff[kMaxCluster + 1];
};

static_assert(offsetof(FusedSmem, chist) % 16 == 0, "uint4 reads of the histograms");
static_assert(offsetof(FusedSmem, scratch) % 16 == 0, "uint4 reads of the bin ends");
static_assert((offsetof(FusedSmem, loc) + offsetof(LocalTopkSmem, sel) +
               offsetof(SelectSmem, hist)) % 16 == 0, "uint4 reads of the coarse histogram");

constexpr int kBinsPerThread = kNB / kNT;   // 2
static_assert(3 * kNB * sizeof(uint32_t) <= sizeof(FusedSmem::chist), "OFF, END, CNT in chist");
static_assert(kScratch >= kGatherCap, "the heavy-tie path gathers into scratch");

__host__ __device__ constexpr size_t fused_dyn_offset() {
  return (sizeof(FusedSmem) + 127) & ~size_t(127);
}

__device__ __forceinline__ ull rank_key(uint32_t k, uint32_t gid) {
  return ((ull)k << 32) | (ull)(~gid);
}

// One digit of the cluster-wide select over `h` (NB bins, PER per thread):
// histogram this CTA's keys, then sum every CTA's histogram for this thread's
// bins and find the bin holding the need-th key (highest bins first).
template <int NB, int PER, typename Visit>
__device__ __forceinline__ void cluster_digit(cg::cluster_group& cluster, int nranks, int need,
                                              uint32_t prefix, uint32_t mask, int shift,
                                              Visit visit, uint32_t* h, FusedSmem& sm) {
  static_assert(NB == PER * kNT, "bins per thread");
  const int tid = threadIdx.x;
  for (int b = tid; b < NB; b += kNT) h[b] = 0u;
  __syncthreads();
  visit([&](uint32_t k) {
    if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & (NB - 1)], 1u);
  });
  cluster.sync();
  const int g = NB - PER * (tid + 1);   // this thread's bins g .. g+PER-1
  int c[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) c[j] = 0;
  for (int rk = 0; rk < nranks; ++rk) {
    const uint32_t* rh = cluster.map_shared_rank(h, rk);
    if constexpr (PER == 4) {
      const uint4 q = *reinterpret_cast<const uint4*>(rh + g);
      c[0] += (int)q.w; c[1] += (int)q.z; c[2] += (int)q.y; c[3] += (int)q.x;
    } else {
      const uint2 q = *reinterpret_cast<const uint2*>(rh + g);
      c[0] += (int)q.y; c[1] += (int)q.x;
    }
  }
  int local = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) local += c[j];
  int total;
  int running = block_exclusive_scan(local, sm.scan, &total);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if (running < need && running + c[j] >= need) {
      sm.bin = g + PER - 1 - j;
      sm.above = running;
      sm.count = c[j];
    }
    running += c[j];
  }
  __syncthreads();
}

// Cluster-wide radix select: the need-th largest key over every CTA's keys
// (visit(f) calls f(k) for each key the calling thread holds).  Every CTA
// computes the same result.  `phase` counts histogram uses across calls: the
// buffer written in a pass was last read remotely two passes earlier, before
// the cluster barrier of the previous pass, so one barrier per digit suffices.
template <typename Visit>
__device__ SelectResult cluster_select(cg::cluster_group& cluster, int nranks, int need,
                                       Visit visit, FusedSmem& sm, int& phase, int pass0 = 0,
                                       uint32_t prefix = 0, uint32_t mask = 0) {
#pragma unroll 1
  for (int pass = pass0; pass < 3; ++pass) {
    uint32_t* h = sm.chist[phase & 1];
    ++phase;
    int shift;
    if (pass < 2) {
      shift = pass == 0 ? 21 : 10;
      cluster_digit<2048, 4>(cluster, nranks, need, prefix, mask, shift, visit, h, sm);
    } else {
      shift = 0;
      cluster_digit<1024, 2>(cluster, nranks, need, prefix, mask, shift, visit, h, sm);
    }
    const int nb = pass < 2 ? 2048 : 1024;
    const int b = sm.bin, above = sm.above, count = sm.count;
    need -= above;
    prefix |= (uint32_t)b << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    if (count == need) return SelectResult{prefix - 1u, 0};
  }
  return SelectResult{prefix, need};
}

// Entries of a descending list that rank above `key` (all keys distinct).
__device__ __forceinline__ int count_above(const ull* list, int len, ull key) {
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (list[mid] > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Descending bitonic sort of NT*E keys, thread t holding indices t*E .. t*E+E-1.
// Partners closer than E are in the thread, closer than 32*E in the warp
// (shuffles), farther ones go through `xchg` (NT*E entries of shared memory).
template <int E>
__device__ __forceinline__ void bitonic_desc(ull (&v)[E], ull* xchg) {
  const int t = threadIdx.x;
  constexpr int P = kNT * E;
#pragma unroll 1
  for (int k = 2; k <= P; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j < E) {
        // partners inside the thread; j is 1 or 2, spelled out so v stays in registers
        if (j == 1) {
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const bool desc = ((t * E + e) & k) == 0;
            const ull a = v[e], b = v[e + 1];
            if ((a < b) == desc) { v[e] = b; v[e + 1] = a; }
          }
        } else if constexpr (E == 4) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool desc = ((t * E + e) & k) == 0;
            const ull a = v[e], b = v[e + 2];
            if ((a < b) == desc) { v[e] = b; v[e + 2] = a; }
          }
        }
      } else if (j < 32 * E) {
        const int lm = j / E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = t * E + e;
          const ull other = __shfl_xor_sync(kFull, v[e], lm);
          const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
          v[e] = keep_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) xchg[t * E + e] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = t * E + e;
          const ull other = xchg[i ^ j];
          const bool keep_max = ((i & j) == 0) == ((i & k) == 0);
          v[e] = keep_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
        }
        __syncthreads();
      }
    }
  }
}

struct FusedArgs {
  const float* logits;
  int64_t ld;
  int rows, S, I, K;
  const int32_t* row_starts;
  const int32_t* row_ends;
  const int32_t* bt;
  int reqs, max_blocks, bs;
  const int32_t* row_to_req;
  int32_t* ids;
  float* scores;
  int32_t* slots;
  int32_t* counts;
  int32_t* local_idx;
  float* cand_out;
  uint32_t* flags;
  int stage_cap;
  ShardMath sh;
  FastDiv fbs;
};

// Slots and global ranks for this CTA's E-per-thread sorted winners.
template <int E>
__device__ __forceinline__ void finish_winners(const FusedArgs& a, cg::cluster_group& cluster,
                                               FusedSmem& sm, int s, int r, int w, int total) {
  const int tid = threadIdx.x;
  ull* win = sm.scratch;
  ull* others = sm.scratch + kMaxK;
  ull v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    v[e] = i < w ? win[i] : 0ull;
  }
  __syncthreads();
  bitonic_desc<E>(v, win);
#pragma unroll
  for (int e = 0; e < E; ++e) win[tid * E + e] = v[e];

  // ---- slots: this shard's winners in rank order, through its block table --
  const int req = a.row_to_req ? a.row_to_req[r] : r;
  const bool req_ok = req >= 0 && req < a.reqs;
  const int32_t* table = a.bt + ((int64_t)s * a.reqs + (req_ok ? req : 0)) * a.max_blocks;
  int32_t* dst = a.slots + ((int64_t)s * a.rows + r) * a.K;
  int blk[E];
  uint32_t off[E];
  bool bad = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    blk[e] = -1;
    off[e] = 0;
    if (tid * E + e < w) {
      const uint32_t l = a.sh.local_slot(~(uint32_t)v[e]);
      const uint32_t col = fdivmod(l, a.fbs, &off[e]);
      if (req_ok && col < (uint32_t)a.max_blocks)
        blk[e] = col < (uint32_t)kTableCap ? sm.sbt[col] : __ldg(table + col);
      else bad = true;
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    if (i < w) {
      const int64_t slot = (int64_t)blk[e] * a.bs + off[e];
      const bool ok = blk[e] >= 0 && slot <= (int64_t)INT32_MAX;
      bad |= !ok;
      dst[i] = ok ? (int32_t)slot : -1;
    }
  }
  for (int i = w + tid; i < a.K; i += kNT) dst[i] = -1;
  if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  if (tid == 0) {
    if (a.counts) a.counts[(int64_t)s * a.rows + r] = w;
    sm.w = w;
  }
  cluster.sync();  // every CTA's sorted winners are published

  // ---- merged ids: rank = own position + other shards' winners above --------
  if (tid < a.S) sm.wr[tid] = *cluster.map_shared_rank(&sm.w, tid);
  __syncthreads();
  if (tid == 0) {
    int o = 0;
    for (int rk = 0; rk < a.S; ++rk) {
      sm.off[rk] = o;
      if (rk != s) o += sm.wr[rk];
    }
  }
  __syncthreads();
  for (int rk = 0; rk < a.S; ++rk) {
    if (rk == s) continue;
    const ull* remote = cluster.map_shared_rank(win, rk);
    const int len = sm.wr[rk], o = sm.off[rk];
    for (int j = tid; j < len; j += kNT)
      if (o + j < kMaxK) others[o + j] = remote[j];
  }
  __syncthreads();
  int32_t* out_ids = a.ids + (int64_t)r * a.K;
  float* out_sc = a.scores ? a.scores + (int64_t)r * a.K : nullptr;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = tid * E + e;
    if (i < w) {
      int rank = i;
      for (int rk = 0; rk < a.S; ++rk)
        if (rk != s) rank += count_above(others + sm.off[rk], sm.wr[rk], v[e]);
      if (rank < a.K) {
        out_ids[rank] = (int32_t)~(uint32_t)v[e];
        if (out_sc) out_sc[rank] = key_score((uint32_t)(v[e] >> 32));
      }
    }
  }
  if (s == 0) {
    for (int j = min(total, a.K) + tid; j < a.K; j += kNT) {
      out_ids[j] = -1;
      if (out_sc) out_sc[j] = -INFINITY;
    }
  }
}

// Merge and convert by one fine histogram (the common case).  Candidates whose
// score key is at least floor_key (no candidate below it can win) are binned by
// bin(x) = (score_key(x) - floor_key) >> sh, highest bin first.  Each CTA
// counting-sorts its binned candidates into bin order, then sorts each (small)
// bin by placing every element at its bin start plus the number of same-bin
// elements ranked above it, and publishes the sorted list LS with the bin
// starts OFF and sizes CNT.  After one cluster barrier every CTA sums the bin
// sizes over the cluster (DSMEM) to find the bin b* holding the K-th
// candidate, copies every other CTA's sorted list down to the end of b*
// (coalesced DSMEM reads, at most K - 1 + kBinCap entries in all), and works
// in its own shared memory: the threshold among b*'s few members; then its
// winner i (LS[i]) has compacted-slot position i and merged-id position
// i + (entries above it in each other CTA's sorted list, by binary search).
// Returns false, before writing any output, when a bin holding winners has
// more than kBinCap candidates (heavy ties); the decision is the same in every
// CTA.  On false the caller must pass a cluster barrier before reusing chist,
// scratch or cand, which other CTAs may still be reading.
__device__ __forceinline__ int fine_bin(ull x, uint32_t floor_key, int sh) {
  return (int)(((uint32_t)(x >> 32) - floor_key) >> sh);
}

__device__ bool merge_by_bins(const FusedArgs& a, cg::cluster_group& cluster, FusedSmem& sm,
                              const ull (&ck)[kCandPerThread], int s, int r, int total,
                              uint32_t floor_key, int sh) {
  const int tid = threadIdx.x;
  const int K = a.K;
  uint32_t* OFF = &sm.chist[0][0];        // bin start in the lists
  uint32_t* END = OFF + kNB;               // fill cursor, then bin end
  uint32_t* CNT = OFF + 2 * kNB;           // bin size (what other CTAs sum)
  ull* LB = sm.scratch;                    // candidates in bin order
  ull* LS = sm.scratch + kMaxK;            // ... sorted (published)
  ull* others = sm.scratch + 2 * kMaxK;    // other CTAs' sorted lists, down to b*
  ull* M = reinterpret_cast<ull*>(sm.loc.sel.hist);

  // Own histogram (END as counters), then the descending-bin exclusive prefix.
  for (int b = tid; b < kNB; b += kNT) END[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kCandPerThread; ++q)
    if (ck[q] && (uint32_t)(ck[q] >> 32) >= floor_key) atomicAdd(&END[fine_bin(ck[q], floor_key, sh)], 1u);
  __syncthreads();
  const int g = kNB - kBinsPerThread * (tid + 1);   // bins g, g+1, taken highest first
  int c[kBinsPerThread];
  int local = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    c[j] = (int)END[g + kBinsPerThread - 1 - j];
    local += c[j];
  }
  int nbin;
  int run = block_exclusive_scan(local, sm.scan, &nbin);
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    const int b = g + kBinsPerThread - 1 - j;
    OFF[b] = (uint32_t)run;
    END[b] = (uint32_t)run;     // becomes the fill cursor, then the bin end
    CNT[b] = (uint32_t)c[j];
    run += c[j];
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kCandPerThread; ++q)
    if (ck[q] && (uint32_t)(ck[q] >> 32) >= floor_key)
      LB[atomicAdd(&END[fine_bin(ck[q], floor_key, sh)], 1u)] = ck[q];
  __syncthreads();
  for (int p = tid; p < nbin; p += kNT) {          // sort within bins
    const ull x = LB[p];
    const int b = fine_bin(x, floor_key, sh);
    int pos = (int)OFF[b];
    for (uint32_t q = OFF[b]; q < END[b]; ++q) pos += LB[q] > x;
    LS[pos] = x;
  }
  cluster.sync();   // every CTA's LS, OFF and CNT are published

  // Global counts of this thread's bins, from the top: the K-th candidate's bin.
  int G[kBinsPerThread];
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) G[j] = 0;
  for (int rk = 0; rk < a.S; ++rk) {
    const uint2 q = *reinterpret_cast<const uint2*>(cluster.map_shared_rank(CNT, rk) + g);
    G[0] += (int)q.y;
    G[1] += (int)q.x;
  }
  local = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) local += G[j];
  if (tid == 0) sm.bstar = 0;        // all binned candidates win when total <= K
  __syncthreads();
  int tot;
  run = block_exclusive_scan(local, sm.scan, &tot);
  int mx = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    const int b = g + kBinsPerThread - 1 - j;
    if (run < K && G[j] > mx) mx = G[j];            // a bin holding winners
    if (total > K && run < K && run + G[j] >= K) {
      sm.bstar = b;
      sm.bneed = K - run;
    }
    run += G[j];
  }
  if (mx > kBinCap) atomicMax(&sm.bmax, mx);
  __syncthreads();
  if (sm.bmax > kBinCap) return false;
  const int bstar = sm.bstar;

  // Copy every other CTA's sorted list down to the end of bin b*.
  if (tid < a.S) {
    const uint32_t o = cluster.map_shared_rank(OFF, tid)[bstar];
    const uint32_t n = cluster.map_shared_rank(CNT, tid)[bstar];
    sm.wr[tid] = (int)(o + n);           // entries in bins >= b*
    sm.moff[tid] = (int)n;               // of which in b*
  }
  __syncthreads();
  // Every thread forms the (at most kMaxCluster) copy offsets itself, and per
  // chunk of kNT positions issues the loads from all ranks before any store:
  // the remote (DSMEM) reads then overlap instead of queueing behind stores.
  int len[kMaxCluster], off[kMaxCluster], maxlen = 0;
  {
    int o = 0;
#pragma unroll
    for (int rk = 0; rk < kMaxCluster; ++rk) {
      len[rk] = (rk < a.S && rk != s) ? sm.wr[rk] : 0;
      off[rk] = o;
      o += len[rk];
      maxlen = max(maxlen, len[rk]);
    }
  }
  if (tid < kMaxCluster) sm.off[tid] = off[tid];
  for (int j0 = 0; j0 < maxlen; j0 += kNT) {
    const int j = j0 + tid;
    ull v[kMaxCluster];
#pragma unroll
    for (int rk = 0; rk < kMaxCluster; ++rk) {
      // Ranks past the cluster map to this CTA (len 0: nothing is read).
      const ull* remote = cluster.map_shared_rank(LS, rk < a.S ? rk : s);
      v[rk] = j < len[rk] ? remote[j] : 0ull;
    }
#pragma unroll
    for (int rk = 0; rk < kMaxCluster; ++rk)
      if (j < len[rk] && off[rk] + j < kMaxK + kBinCap) others[off[rk] + j] = v[rk];
  }
  __syncthreads();

  // The K-th candidate's rank key: winners are the keys >= thr.
  ull thr = 1ull;                                   // all candidates (keys are > 0)
  if (total > K) {
    const int warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
      int o = 0;
      for (int rk = 0; rk < a.S; ++rk) {
        sm.rk_m[rk] = o;                 // where rank rk's members go in M
        o += sm.moff[rk];
      }
      sm.total = o;
    }
    __syncthreads();
    if (warp < a.S) {     // b*'s members: the tail of every CTA's (copied) list
      const ull* src = warp == s ? LS + OFF[bstar]
                                 : others + sm.off[warp] + sm.wr[warp] - sm.moff[warp];
      for (int j = lane; j < sm.moff[warp]; j += 32) M[sm.rk_m[warp] + j] = src[j];
    }
    __syncthreads();
    const int nm = sm.total, need = sm.bneed;
    if (tid < nm) {
      const ull x = M[tid];
      int above = 0;
      for (int j = 0; j < nm; ++j) above += M[j] > x;
      if (above == need - 1) sm.thr64 = x;
    }
    __syncthreads();
    thr = sm.thr64;
  }

  // Winner i of this CTA is LS[i]: compacted-slot position i; merged-id
  // position i + the entries above it in every other CTA's sorted list.
  int nmine = 0;
  for (int i = tid; i < nbin; i += kNT) nmine += LS[i] >= thr;
  nmine = __reduce_add_sync(kFull, nmine);
  if ((tid & 31) == 0 && nmine) atomicAdd(&sm.nown, nmine);
  __syncthreads();
  const int w = min(sm.nown, K);
  const int req = a.row_to_req ? a.row_to_req[r] : r;
  const bool req_ok = req >= 0 && req < a.reqs;
  const int32_t* table = a.bt + ((int64_t)s * a.reqs + (req_ok ? req : 0)) * a.max_blocks;
  int32_t* dst = a.slots + ((int64_t)s * a.rows + r) * K;
  int32_t* out_ids = a.ids + (int64_t)r * K;
  float* out_sc = a.scores ? a.scores + (int64_t)r * K : nullptr;
  int blk[kCandPerThread];
  uint32_t boff[kCandPerThread];
  bool bad = false;
#pragma unroll
  for (int u = 0; u < kCandPerThread; ++u) {     // every table load first
    const int i = tid + u * kNT;
    blk[u] = -1;
    boff[u] = 0;
    if (i < w) {
      const uint32_t l = a.sh.local_slot(~(uint32_t)LS[i]);
      const uint32_t col = fdivmod(l, a.fbs, &boff[u]);
      if (req_ok && col < (uint32_t)a.max_blocks)
        blk[u] = col < (uint32_t)kTableCap ? sm.sbt[col] : __ldg(table + col);
      else bad = true;
    }
  }
#pragma unroll
  for (int u = 0; u < kCandPerThread; ++u) {
    const int i = tid + u * kNT;
    if (i < K) {
      int32_t v = -1;
      if (i < w) {
        const ull x = LS[i];
        int grank = i;
        for (int rk = 0; rk < a.S; ++rk)
          if (rk != s) grank += count_above(others + sm.off[rk], sm.wr[rk], x);
        const int64_t slot = (int64_t)blk[u] * a.bs + boff[u];
        const bool ok = blk[u] >= 0 && slot <= (int64_t)INT32_MAX;
        bad |= !ok;
        v = ok ? (int32_t)slot : -1;
        if (grank < K) {
          out_ids[grank] = (int32_t)~(uint32_t)x;
          if (out_sc) out_sc[grank] = key_score((uint32_t)(x >> 32));
        }
      }
      dst[i] = v;
    }
  }
  if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);
  if (tid == 0 && a.counts) a.counts[(int64_t)s * a.rows + r] = w;
  if (s == 0) {
    for (int j = min(total, K) + tid; j < K; j += kNT) {
      out_ids[j] = -1;
      if (out_sc) out_sc[j] = -INFINITY;
    }
  }
  return true;
}

__global__ void __launch_bounds__(kNT, 2) fused_kernel(const FusedArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FusedSmem& sm = *reinterpret_cast<FusedSmem*>(smem_raw);
  float* stage = reinterpret_cast<float*>(smem_raw + fused_dyn_offset());
  const int tid = threadIdx.x, lane = tid & 31;
  const int s = (int)cluster.block_rank();
  const int r = blockIdx.x / a.S;
  const int K = a.K;
  const float* row = a.logits + ((int64_t)s * a.rows + r) * a.ld;

  // ---- this shard's local range ------------------------------------------
  int64_t st = a.row_starts ? (int64_t)a.row_starts[r] : 0, en = a.row_ends[r];
  bool bad = false;
  if (st < 0) { st = 0; bad = true; }
  if (en < st) { en = st; bad = true; }
  // st and en are int32 row bounds clamped to >= 0: the 32-bit map applies.
  int64_t lo = a.sh.local_len((uint32_t)st, s), hi = a.sh.local_len((uint32_t)en, s);
  if (hi > a.ld) { hi = a.ld; bad = true; }
  if (lo > hi) { lo = hi; bad = true; }
  const int n = (int)(hi - lo);
  if (tid == 0) {
    if (bad) raise_flag(a.flags, DSA_FLAG_BOUNDS);
    sm.m = min(n, K);
    sm.tied = 0;
    sm.nwin = 0;
    sm.ncl = 0;
    sm.es.nout = 0;
    sm.kmin = 0xffffffffu;
    sm.kmax = 0u;
    sm.bmax = 0;
    sm.nown = 0;
  }
  int32_t* out_idx = a.local_idx ? a.local_idx + ((int64_t)s * a.rows + r) * K : nullptr;
  float2* out_cand = a.cand_out ? reinterpret_cast<float2*>(a.cand_out) + ((int64_t)r * a.S + s) * K
                                : nullptr;
  const bool ordered = out_idx || out_cand;   // intermediates are written in slot order
  // Rows on the register path issue their logit loads first, so that they
  // are in flight during the block-table fetch below.
  const int64_t base = lo & ~int64_t(3);
  const bool reg_path = n > K && hi - base <= RT::kCap;
  float4 v[kVec];
  if (reg_path) {
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int64_t e0 = base + ((int64_t)j * kNT + tid) * 4;
      v[j] = e0 < hi ? __ldg(reinterpret_cast<const float4*>(row + e0))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  {
    // This shard's block-table row, copied asynchronously now so the slot
    // conversion at the end does not wait on it; completed before the barrier
    // that ends the local top-K.  The barriers inside the local top-K order
    // thread 0's initialisation above before any use.
    const int req = a.row_to_req ? a.row_to_req[r] : r;
    if (req >= 0 && req < a.reqs) {
      const int32_t* table = a.bt + ((int64_t)s * a.reqs + req) * a.max_blocks;
      const int ncol = min(a.max_blocks, kTableCap);
      for (int c = tid; c < ncol; c += kNT) cp_async4(&sm.sbt[c], table + c);
    }
  }

  // ---- a1 + a2: local top-K, kept as rank keys -----------------------------
  if (n <= K) {
    for (int j = tid; j < K; j += kNT) {
      if (j < n) {
        const uint32_t l = (uint32_t)(lo + j);
        const float v = row[l];
        const uint32_t gid = a.sh.global_id(s, l);
        sm.cand[j] = rank_key(score_key(v), gid);
        if (out_idx) out_idx[j] = (int32_t)l;
        if (out_cand) out_cand[j] = make_float2(v, __int_as_float((int)gid));
      } else {
        if (out_idx) out_idx[j] = -1;
        if (out_cand) out_cand[j] = make_float2(-INFINITY, __int_as_float(-1));
      }
    }
  } else if (reg_path) {
    uint32_t key[kVec][4];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int64_t e0 = base + ((int64_t)j * kNT + tid) * 4;
      const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) key[j][c] = (e0 + c >= lo && e0 + c < hi) ? score_key(f[c]) : 0u;
    }
    int eq;
    const SelectResult res = select_regs<kNT, kVec>(key, K, sm.loc.sel,
                                                    reinterpret_cast<uint32_t*>(sm.scratch),
                                                    sm.es, &eq);
    // Winners are staged as (score key, slot) words in the scratch area (the
    // select's list is dead by now), then turned into rank keys and written
    // out by all threads together: the per-winner work runs with full warps.
    uint32_t* stage_k = reinterpret_cast<uint32_t*>(sm.scratch);
    uint32_t* stage_l = stage_k + kMaxK;
    auto put = [&](int p, int e, uint32_t k) {
      if (p >= K) return;
      stage_k[p] = k;
      stage_l[p] = (uint32_t)(base + e);
    };
    if (!ordered && (res.take_eq == 0 || res.take_eq == eq))
      emit_unordered<kNT, kVec>(key, res.take_eq == 0 ? res.thr + 1u : res.thr, sm.es, put);
    else
      emit_winners<kNT, kVec>(key, res.thr, res.take_eq, sm.es, put);
    __syncthreads();
    for (int p = tid; p < K; p += kNT) {
      const uint32_t k = stage_k[p], l = stage_l[p];
      const uint32_t gid = a.sh.global_id(s, l);
      sm.cand[p] = rank_key(k, gid);
      if (out_idx) out_idx[p] = (int32_t)l;
      // A zero key stands for both zeros: read the value back for its sign.
      if (out_cand)
        out_cand[p] = make_float2(k == 0x80000000u ? row[l] : key_score(k),
                                  __int_as_float((int)gid));
    }
  } else {
    bool ok;
    const float* data = stage_local_range(row, lo, hi, stage, a.stage_cap, sm.loc, a.flags, &ok);
    local_topk_emit<kNT>(data, n, K, sm.loc, [&](int p, int i, float v) {
      const uint32_t l = (uint32_t)(lo + i);
      const uint32_t gid = a.sh.global_id(s, l);
      sm.cand[p] = rank_key(score_key(v), gid);
      if (out_idx) out_idx[p] = (int32_t)l;
      if (out_cand) out_cand[p] = make_float2(v, __int_as_float((int)gid));
    });
  }
  cp_async_wait_all();   // this thread's block-table words; the barrier publishes them
  __syncthreads();
  const int m = sm.m;
  ull ck[kCandPerThread];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < kCandPerThread; ++q) {
    const int i = tid + q * kNT;
    ck[q] = i < m ? sm.cand[i] : 0ull;    // 0: no candidate (valid keys are > 0)
    if (ck[q]) {
      kmin = min(kmin, (uint32_t)(ck[q] >> 32));
      kmax = max(kmax, (uint32_t)(ck[q] >> 32));
    }
  }
  kmin = __reduce_min_sync(kFull, kmin);
  kmax = __reduce_max_sync(kFull, kmax);
  if (lane == 0) {
    atomicMin(&sm.kmin, kmin);
    atomicMax(&sm.kmax, kmax);
  }
  // Coarse histogram (one bin per binade: top 9 key bits) of this CTA's
  // candidates: summed over the cluster it locates the binade of the K-th
  // candidate, the floor of the fine bins.
  uint32_t* coarse = sm.loc.sel.hist;
  for (int b = tid; b < kCoarse; b += kNT) coarse[b] = 0u;
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kCandPerThread; ++q)
    if (ck[q]) atomicAdd(&coarse[(uint32_t)(ck[q] >> 55)], 1u);
  cluster.sync();  // every CTA's candidates are in place

  // ---- a3 + a4: global winners, their ranks and this shard's slots ---------
  if (tid < a.S) {
    sm.rk_m[tid] = *cluster.map_shared_rank(&sm.m, tid);
    sm.rk_min[tid] = *cluster.map_shared_rank(&sm.kmin, tid);
    sm.rk_max[tid] = *cluster.map_shared_rank(&sm.kmax, tid);
  }
  __syncthreads();
  int total = 0;
  uint32_t gmin = 0xffffffffu, gmax = 0u;
  for (int rk = 0; rk < a.S; ++rk) {
    total += sm.rk_m[rk];
    gmin = min(gmin, sm.rk_min[rk]);
    gmax = max(gmax, sm.rk_max[rk]);
  }
  if (total == 0) {   // every shard is empty
    int32_t* dst = a.slots + ((int64_t)s * a.rows + r) * K;
    for (int i = tid; i < K; i += kNT) dst[i] = -1;
    if (tid == 0 && a.counts) a.counts[(int64_t)s * a.rows + r] = 0;
    if (s == 0)
      for (int j = tid; j < K; j += kNT) {
        a.ids[(int64_t)r * K + j] = -1;
        if (a.scores) a.scores[(int64_t)r * K + j] = -INFINITY;
      }
    cluster.sync();
    return;
  }
  uint32_t floor_key = gmin;
  if (total > K) {
    static_assert(kCoarse == kNT, "one coarse bin per thread");
    const int gc = kCoarse - 1 - tid;       // bins from the top
    int c = 0;
    for (int rk = 0; rk < a.S; ++rk) c += (int)cluster.map_shared_rank(coarse, rk)[gc];
    int tot;
    const int run = block_exclusive_scan(c, sm.scan, &tot);
    if (run < K && run + c >= K) sm.bin = gc;
    __syncthreads();
    floor_key = max(gmin, (uint32_t)sm.bin << 23);
  }
  int sh = 0;
  while (((gmax - floor_key) >> sh) >= (uint32_t)kNB) ++sh;
  if (merge_by_bins(a, cluster, sm, ck, s, r, total, floor_key, sh)) {
    cluster.sync();  // no CTA leaves while another still reads its shared memory
    return;
  }
  cluster.sync();    // other CTAs are done reading this CTA's bins

  // ---- heavy ties: select across the cluster, then sort ---------------------
  const bool all = total <= K;
  bool tie = false;
  uint32_t thr1 = 0, thr2 = 0;
  int phase = 0;
  if (!all) {
    auto visit1 = [&](auto&& f) {
#pragma unroll
      for (int q = 0; q < kCandPerThread; ++q)
        if (ck[q]) f((uint32_t)(ck[q] >> 32));
    };
    // First digit across the cluster.
    uint32_t* h = sm.chist[phase & 1];
    ++phase;
    cluster_digit<2048, 4>(cluster, a.S, K, 0u, 0u, 21, visit1, h, sm);
    const uint32_t b1 = (uint32_t)sm.bin;
    const int count1 = sm.count, need = K - sm.above;
    const uint32_t prefix = b1 << 21, mask = 0x7ffu << 21;
    if (count1 == need) {
      thr1 = prefix - 1u;                              // the whole bin is in
    } else if (count1 <= kGatherCap) {
      // Publish this CTA's threshold-bin candidates (in place of its candidate
      // list, which the registers now hold), then gather everyone's.
      int mine = 0;
#pragma unroll
      for (int q = 0; q < kCandPerThread; ++q)
        mine += ck[q] && ((uint32_t)(ck[q] >> 32) & mask) == prefix;
      const int incl = warp_inclusive_scan(mine);
      int wb = 0;
      if (lane == 31 && incl) wb = atomicAdd(&sm.ncl, incl);
      int p = __shfl_sync(kFull, wb, 31) + incl - mine;
#pragma unroll
      for (int q = 0; q < kCandPerThread; ++q)
        if (ck[q] && ((uint32_t)(ck[q] >> 32) & mask) == prefix) sm.cand[p++] = ck[q];
      cluster.sync();
      if (tid < a.S) sm.wr[tid] = *cluster.map_shared_rank(&sm.ncl, tid);
      __syncthreads();
      ull* g = sm.scratch;
      int o = 0;
      for (int rk = 0; rk < a.S; ++rk) {
        const ull* remote = cluster.map_shared_rank(sm.cand, rk);
        const int len = sm.wr[rk];
        for (int j = tid; j < len; j += kNT)
          if (o + j < kGatherCap) g[o + j] = remote[j];
        o += len;
      }
      __syncthreads();
      const int ng = min(o, kGatherCap);
      auto visitg = [&](auto&& f) {
        for (int i = tid; i < ng; i += kNT) f((uint32_t)(g[i] >> 32));
      };
      int eq;
      const SelectResult a2 = radix_select_from<kNT>(1, prefix, mask, need, visitg, sm.loc.sel,
                                                     &eq);
      thr1 = a2.thr;
      if (a2.take_eq > 0) {
        if (eq > a2.take_eq) {
          auto visit2 = [&](auto&& f) {
            for (int i = tid; i < ng; i += kNT)
              if ((uint32_t)(g[i] >> 32) == thr1) f((uint32_t)g[i]);
          };
          int eq2;
          const SelectResult b = radix_select_from<kNT>(0, 0u, 0u, a2.take_eq, visit2, sm.loc.sel,
                                                        &eq2);
          thr2 = b.take_eq > 0 ? b.thr : b.thr + 1u;   // ~id >= thr2: the smallest ids
          tie = true;
        } else {
          thr1 -= 1u;                                  // the whole tied group is in
        }
      }
    } else {
      // A huge threshold bin: finish the select digit by digit across the cluster.
      const SelectResult a1 = cluster_select(cluster, a.S, need, visit1, sm, phase, 1, prefix,
                                             mask);
      thr1 = a1.thr;
      if (a1.take_eq > 0) {
        int e = 0;
#pragma unroll
        for (int q = 0; q < kCandPerThread; ++q) e += ck[q] && (uint32_t)(ck[q] >> 32) == thr1;
        e = __reduce_add_sync(kFull, e);
        if (lane == 0 && e) atomicAdd(&sm.tied, e);
        cluster.sync();
        int tied = 0;
        for (int rk = 0; rk < a.S; ++rk) tied += *cluster.map_shared_rank(&sm.tied, rk);
        if (tied > a1.take_eq) {
          auto visit2 = [&](auto&& f) {
#pragma unroll
            for (int q = 0; q < kCandPerThread; ++q)
              if (ck[q] && (uint32_t)(ck[q] >> 32) == thr1) f((uint32_t)ck[q]);
          };
          const SelectResult b = cluster_select(cluster, a.S, a1.take_eq, visit2, sm, phase);
          thr2 = b.take_eq > 0 ? b.thr : b.thr + 1u;
          tie = true;
        } else {
          thr1 -= 1u;
        }
      }
    }
  }
  __syncthreads();   // the gathered list in scratch is no longer read

  // This CTA's winners, gathered in any order.
  ull* win = sm.scratch;
#pragma unroll
  for (int q = 0; q < kCandPerThread; ++q) {
    bool wsel = false;
    if (ck[q]) {
      const uint32_t k1 = (uint32_t)(ck[q] >> 32);
      wsel = all || k1 > thr1 || (tie && k1 == thr1 && (uint32_t)ck[q] >= thr2);
    }
    const unsigned msk = __ballot_sync(kFull, wsel);
    int wbase = 0;
    if (lane == 0 && msk) wbase = atomicAdd(&sm.nwin, __popc(msk));
    wbase = __shfl_sync(kFull, wbase, 0);
    const int slot = wbase + __popc(msk & lanemask_lt());
    if (wsel && slot < kMaxK) win[slot] = ck[q];
  }
  __syncthreads();
  const int w = min(sm.nwin, K);
  if (w <= kNT) finish_winners<1>(a, cluster, sm, s, r, w, total);
  else if (w <= 2 * kNT) finish_winners<2>(a, cluster, sm, s, r, w, total);
  else finish_winners<4>(a, cluster, sm, s, r, w, total);
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
  if (ld > (int64_t)INT32_MAX || (int64_t)rows * S > (int64_t)INT32_MAX ||
      (int64_t)I * S > (int64_t)INT32_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!logits || !row_ends || !block_table || !ids || !slots || !aligned16(logits))
    return DSA_ERR_INVALID_ARG;
  if (cand && !aligned16(cand)) return DSA_ERR_INVALID_ARG;
  // Rows that fit the register path need no staging area; otherwise stage as
  // much as the device's per-block shared memory allows (longer rows are read
  // from global memory).
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  const size_t fixed = fused_dyn_offset();
  if ((size_t)optin < fixed) return DSA_ERR_UNSUPPORTED;
  const int64_t room = (int64_t)(((size_t)optin - fixed) / sizeof(float)) & ~int64_t(3);
  int stage_cap = 0;
  if (ld > RT::kCap) stage_cap = (int)min(min(ld, room), (int64_t)kStageCapElems);
  const size_t smem = fixed + (size_t)stage_cap * sizeof(float);
  if (cudaFuncSetAttribute(fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  FusedArgs args{logits, ld, rows, S, I, K, row_starts, row_ends, block_table, reqs, max_blocks,
                 block_size, row_to_req, ids, scores, slots, counts, local_idx, cand, err_flags,
                 stage_cap, ShardMath(S, I), FastDiv((uint32_t)block_size)};
  const cudaError_t e = launch_kernel(fused_kernel, dim3((unsigned)(rows * S)), dim3(kNT), smem,
                                      stream, (unsigned)S, args);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
