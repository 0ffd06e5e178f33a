"""Sparse-indexer top-K under DCP, step by step.  Test infrastructure.

Sources (page titles and sections):
  [P46076] PR #46076 report, "[Attention][DSA] support dcp for
           FLASHINFER_MLA_SPARSE": section 实现拆解 (implementation breakdown)
           items 1, 2 and 4; section 关键源码片段 (key source snippets), the
           `_merge_dcp_topk_global` docstring and the packed-buffer allocation;
           section 评论区精华 (review highlights), "compact valid slots fused
           into the convert kernel".
  [P40996] PR #40996 report, "DCP supports hybrid attention": section 关键源码片段,
           `AttentionSpec.max_num_blocks_per_req` (rank-local paged block tables).

Readings taken where the pages are silent (listed with the rest in the design
notes):
  * ranking: score descending, ties to the smaller global token id; -0.0 and
    +0.0 are the same score; -inf inside a row's range is a real score that
    ranks above padding; inputs hold no NaN (asserted);
  * a shard's top-K list is written in ascending local slot order, -1 padded;
  * the merged list is written in rank order, -1 padded;
  * the id lane of a packed candidate holds the int32 id's bit pattern;
  * local indices are absolute local slots (every recipe has row_start = 0);
  * compacted slots keep merged-list order (the pages' atomics leave it open).

Padding in outputs: ids/slots -1, scores -inf.
"""
from __future__ import annotations

import numpy as np

from . import dcp_layout


def _scores(v) -> np.ndarray:
    """fp64 copy of fp32 scores with -0.0 folded into +0.0 (same score)."""
    v = np.asarray(v, np.float64) + 0.0
    assert not np.isnan(v).any(), "NaN scores are outside the method's domain"
    return v


def rank_order(scores, ids) -> np.ndarray:
    """Permutation listing entries by score descending, then id ascending."""
    return np.lexsort((np.asarray(ids, np.int64), -_scores(scores)))


def global_topk(x_row, start: int, end: int, K: int):
    """The definition the sharded path must reproduce [P46076 item 1]: the K
    best tokens of the global range [start, end), best first.

    Returns (ids int64[K], scores float32[K]); -1 / -inf after min(K, end-start).
    """
    t = np.arange(start, end, dtype=np.int64)
    v = np.asarray(x_row[start:end], np.float32)
    take = rank_order(v, t)[:K]
    ids = np.full(K, -1, np.int64)
    sc = np.full(K, -np.inf, np.float32)
    ids[:len(take)] = t[take]
    sc[:len(take)] = v[take]
    return ids, sc


def shard_topk(local_row, lo: int, hi: int, K: int) -> np.ndarray:
    """One shard's local top-K over its local slots [lo, hi) [P46076 snippet:
    "topk_indices are top-K positions in this rank's local KV shard"].

    Within a shard, local slot order is global id order, so ties go to the
    smaller slot.  Output: chosen slots ascending, then -1.  int64[K].
    """
    l = np.arange(lo, hi, dtype=np.int64)
    v = np.asarray(local_row[lo:hi], np.float32)
    chosen = np.sort(l[rank_order(v, l)[:K]])
    out = np.full(K, -1, np.int64)
    out[:len(chosen)] = chosen
    return out


def pack(local_row, local_idx, s: int, S: int, I: int):
    """(score, global id) candidates of one shard's top-K [P46076 item 1 and the
    `packed` [batch, topk, 2] fp32 buffer in the snippet].

    A valid local slot l becomes (local_row[l], global id of slot l of shard s);
    padding (-1) becomes (-inf, -1).  Returns (scores float32[K], ids int64[K]).
    """
    local_idx = np.asarray(local_idx, np.int64)
    valid = local_idx >= 0
    sc = np.full(local_idx.shape, -np.inf, np.float32)
    ids = np.full(local_idx.shape, -1, np.int64)
    sc[valid] = np.asarray(local_row, np.float32)[local_idx[valid]]
    if valid.any():
        ids[valid] = dcp_layout.local_to_global(s, local_idx[valid], S, I)
    return sc, ids


def merge(cand_scores, cand_ids, K: int):
    """Stable global top-K of gathered candidates [P46076 item 1,
    `stable_topk_from_gathered_candidates_cutedsl`, and the docstring: the
    result overwrites topk_indices with global token ids, -1 for padding].

    Candidates with id < 0 are padding and never selected.  Returns
    (ids int64[K], scores float32[K]) best first.
    """
    cand_ids = np.asarray(cand_ids, np.int64)
    valid = cand_ids >= 0
    v = np.asarray(cand_scores, np.float32)[valid]
    t = cand_ids[valid]
    take = rank_order(v, t)[:K]
    ids = np.full(K, -1, np.int64)
    sc = np.full(K, -np.inf, np.float32)
    ids[:len(take)] = t[take]
    sc[:len(take)] = v[take]
    return ids, sc


def convert_compact(ids, S: int, I: int, tables, block_size: int):
    """Global ids -> every shard's physical KV slots, valid ones first [P46076
    item 4, `_convert_req_index_to_global_index_kernel` with DCP de-interleave
    and the COMPACT_TO_FRONT branch; P40996 rank-local block tables].

    `tables` [S, max_blocks] holds each shard's block-table row for this query
    row's request.  For each shard s, walk the merged ids in order; an id held
    by s at local slot l maps to tables[s, l // block_size] * block_size +
    l % block_size and is appended.  Ids of other shards and -1 are skipped.  A
    slot whose block column lies outside the table, or whose table entry is
    negative, is appended as -1 and flags an error.

    Returns (slots int64[S, K], counts int64[S], error bool).
    """
    ids = np.asarray(ids, np.int64)
    tables = np.asarray(tables, np.int64)
    K = ids.shape[0]
    valid = ids >= 0
    shard = np.full(K, -1, np.int64)
    local = np.full(K, -1, np.int64)
    if valid.any():
        shard[valid], local[valid] = dcp_layout.global_to_local(ids[valid], S, I)
    out = np.full((S, K), -1, np.int64)
    counts = np.zeros(S, np.int64)
    error = False
    for s in range(S):
        l = local[valid & (shard == s)]          # merged order is kept
        col = l // block_size
        inside = col < tables.shape[1]
        block = np.full(l.shape, -1, np.int64)
        block[inside] = tables[s, col[inside]]
        ok = block >= 0
        slots = np.where(ok, block * block_size + l % block_size, -1)
        error |= bool((~ok).any())
        out[s, :len(slots)] = slots
        counts[s] = len(slots)
    return out, counts, error
