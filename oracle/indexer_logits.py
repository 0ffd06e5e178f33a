"""Indexer logits of the sparse-attention indexer, in fp64.  Test infrastructure.

Sources (page titles and sections):
  [P46076] PR #46076 report, "[Attention][DSA] support dcp for
           FLASHINFER_MLA_SPARSE": section 关键源码片段 (key source snippets),
           `_assert_cutedsl_dcp_merge_supported` (the indexer's `logits` reach
           the DCP top-K as fp32, one row per query token) and the
           `_merge_dcp_topk_global` docstring (each rank scores the tokens of
           its own local KV shard).
  [P52046] PR #52046 report, "DSV3.2 PCP sharding": section 关键源码片段
           (`_sparse_indexer_and_attn`: the indexer scores the cached keys of a
           request before the sparse attention reads the selected ones).

The pages name the step and the type of its output but print no formula.  The
reading taken (listed with the others in the design notes) is the plainest one
for a DeepSeek-V3.2-style sparse-attention indexer: a query token t carries
H_I query heads q[t, h] (d_I values each) and one weight w[t, h] per head; the
indexer key cache holds one key k[u] (d_I values) per token u; the logit is

    logit[t, u] = sum_h  w[t, h] * max(0, q[t, h] . k[u]),

a ReLU of each head's dot product, weighted and summed over the heads.  Queries
and keys are fp8 (e4m3) values, the weights fp32; the oracle decodes the fp8
codes exactly (`e4m3_to_f64`, from the format's definition) and works in fp64.
With DCP, shard s holds the keys of the tokens it owns, in a paged cache
addressed through its block table, and scores its local slots only.
"""
from __future__ import annotations

import numpy as np

from oracle import dcp_layout as OL

IDX_HEADS, IDX_DIM = 64, 128


def e4m3_to_f64(codes) -> np.ndarray:
    """Values of fp8 e4m3 codes (OCP 8-bit floating point, E4M3): sign bit, four
    exponent bits with bias 7, three mantissa bits; exponent field 0 holds the
    subnormals m/8 * 2^-6; the all-ones code S.1111.111 is NaN (there is no
    infinity)."""
    b = np.asarray(codes, np.uint8).astype(np.int64)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = s * val
    return np.where((e == 15) & (m == 7), np.nan, val)


def logits(q, w, keys) -> np.ndarray:
    """One query token against a set of keys.

    q     [H, d] fp64 (decoded query heads)
    w     [H] fp64 head weights
    keys  [n, d] fp64 (decoded keys)
    Returns [n] fp64: sum_h w[h] * max(0, q[h] . key).
    """
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    w = np.asarray(w, np.float64)
    dots = q @ keys.T                                  # [H, n]
    return w @ np.maximum(dots, 0.0)


def shard_logits(q_codes, w, k_codes, starts, ends, S: int, I: int, tables, block_size: int,
                 row_to_req=None, ld: int | None = None, rows=None, fill=np.nan) -> np.ndarray:
    """Each shard's logits of each row's local range, in the layout the shard
    top-K reads.

    q_codes   [R, H, d] uint8 e4m3 query heads; w [R, H] float32 weights
    k_codes   [S, n_slots, d] uint8 e4m3: shard s's key of the token stored at
              physical slot p (block * block_size + offset)
    starts, ends  [R] global [start, end) of each row
    tables    [S, reqs, max_blocks] int32 block tables; row_to_req [R] or None
    Returns [S, len(rows), ld] fp64: entry l of shard s, row r is the logit of
    the token at shard s's local slot l, for l in [n_s(start), n_s(end));
    `fill` elsewhere.  Local slot l of a request lives at physical slot
    tables[s][req][l // block_size] * block_size + l % block_size.
    """
    q_codes = np.asarray(q_codes, np.uint8)
    R = q_codes.shape[0]
    rows = np.arange(R) if rows is None else np.asarray(rows)
    k_codes = np.asarray(k_codes, np.uint8)
    if ld is None:
        ld = max(OL.local_count(int(e), s, S, I) for s in range(S) for e in ends)
    out = np.full((S, len(rows), ld), fill, np.float64)
    for j, r in enumerate(rows):
        q = e4m3_to_f64(q_codes[r])
        req = r if row_to_req is None else int(row_to_req[r])
        for s in range(S):
            lo = OL.local_count(int(starts[r]), s, S, I)
            hi = OL.local_count(int(ends[r]), s, S, I)
            if hi <= lo:
                continue
            l = np.arange(lo, hi)
            phys = tables[s, req, l // block_size].astype(np.int64) * block_size + l % block_size
            out[s, j, lo:hi] = logits(q, w[r], e4m3_to_f64(k_codes[s, phys]))
    return out


def magnitude(q_codes, w, k_codes, starts, ends, S: int, I: int, tables, block_size: int,
              row_to_req=None, ld: int | None = None, rows=None) -> np.ndarray:
    """The same layout, holding sum_h |w[h]| * sum_d |q[h, d] * k[d]|: the scale
    of the rounding error of any evaluation order (the tolerance's unit)."""
    k_abs = np.asarray(k_codes, np.uint8) & np.uint8(0x7F)    # clear the sign bits
    q_abs = np.asarray(q_codes, np.uint8) & np.uint8(0x7F)
    return shard_logits(q_abs, np.abs(np.asarray(w, np.float64)), k_abs, starts, ends, S, I,
                        tables, block_size, row_to_req=row_to_req, ld=ld, rows=rows, fill=0.0)
