"""Sparse MLA decode attention of one shard over its selected KV slots, in fp64.
Test infrastructure.

Sources (page titles and sections):
  [P52046] PR #52046 report, "DSV3.2 PCP sharding": section 关键源码片段 (key
           source snippets), `_fused_norm_rope_kernel` (a cache row is the
           normed latent kv_c followed by the roped k_pe at its tail) and
           `_sparse_indexer_and_attn` (the MQA query is the concatenation of its
           parts on the last dimension; `forward_mqa(q, kv_cache, ...)` returns
           the shard's output and its LSE, which `dcp_manager.combine` merges).
  [P46076] PR #46076 report, "[Attention][DSA] support dcp for
           FLASHINFER_MLA_SPARSE": section 实现拆解 (implementation breakdown)
           item 5 (the sparse MLA decode kernel returns its LSE in base 2,
           `lse_base_on_e = False`), item 4 (the compacted slots it reads).

The attention itself is the softmax definition, written out: with the selected
cache rows k_j (d_qk values each, the first d_v of which are the latent kv_c
and serve as the value v_j),

    s_j = scale * (q . k_j),   O = sum_j exp(s_j) v_j / sum_j exp(s_j),
    lse2 = log2 sum_j exp(s_j).

Readings taken where the pages are silent (listed with the rest in the design
notes): the value of a row is its latent part (the first d_v entries); scale
is a parameter; a shard with no selected slot gives O = 0 and lse2 = -inf (the
combine's empty-shard convention).
"""
from __future__ import annotations

import numpy as np

LN2 = np.log(2.0)


def sparse_mla_decode(q, rows, scale: float, d_v: int):
    """One query (all heads) against the selected cache rows of one shard.

    q     [H, d_qk] fp64
    rows  [n, d_qk] fp64, the cache rows at the shard's selected slots
    Returns (O [H, d_v] fp64, lse2 [H] fp64 base 2).
    """
    q = np.asarray(q, np.float64)
    rows = np.asarray(rows, np.float64)
    H = q.shape[0]
    if rows.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    s = scale * (q @ rows.T)                       # [H, n]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    l = w.sum(axis=1)
    out = (w @ rows[:, :d_v]) / l[:, None]
    lse2 = (m[:, 0] + np.log(l)) / LN2
    return out, lse2


def shard_attention(q, cache, slots, counts, scale: float, d_v: int):
    """Every (shard, row) pair: row r's query against shard s's compacted slots.

    q       [rows, H, d_qk] fp64
    cache   [S, n_slots, d_qk] fp64, each shard's paged KV cache by slot
    slots   [S, rows, K] int, the compacted slots of the read-side conversion
    counts  [S, rows] int, how many of them are valid
    Returns (O [S, rows, H, d_v] fp64, lse2 [S, rows, H] fp64).
    """
    q = np.asarray(q, np.float64)
    S, R = np.asarray(counts).shape
    H = q.shape[1]
    out = np.zeros((S, R, H, d_v))
    lse2 = np.full((S, R, H), -np.inf)
    for s in range(S):
        for r in range(R):
            sel = np.asarray(slots[s][r][:int(counts[s][r])], np.int64)
            out[s, r], lse2[s, r] = sparse_mla_decode(q[r], cache[s][sel], scale, d_v)
    return out, lse2
