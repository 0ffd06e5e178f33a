"""The oracle's steps chained over a workload's rows.  Test infrastructure.

The order is the one `_merge_dcp_topk_global` runs per step in the PR #46076
report ("[Attention][DSA] support dcp for FLASHINFER_MLA_SPARSE", section 关键源码
片段): local top-K on every rank, pack, all_gather along the candidate axis
(here: each shard's slice of one [rows, S*K] buffer), stable merge; then the
convert of section 实现拆解 item 4.
"""
from __future__ import annotations

import numpy as np

from . import dcp_layout, indexer


def run_rows(local_logits, row_starts, row_ends, S: int, I: int, K: int,
             rows=None, tables=None, row_to_req=None, block_size: int = 64):
    """Run shard_topk -> pack -> merge (-> convert) for the listed rows.

    local_logits [S, R, ld] fp32 (per-shard layout), row_starts/row_ends [R]
    global ranges.  tables [S, reqs, max_blocks] enables the convert step.
    Returns a dict of arrays indexed by position in `rows`.
    """
    R = local_logits.shape[1]
    rows = np.arange(R) if rows is None else np.asarray(rows)
    n = len(rows)
    local_idx = np.full((S, n, K), -1, np.int64)
    cand_sc = np.full((n, S * K), -np.inf, np.float32)
    cand_id = np.full((n, S * K), -1, np.int64)
    ids = np.full((n, K), -1, np.int64)
    scores = np.full((n, K), -np.inf, np.float32)
    for j, r in enumerate(rows):
        st, en = int(row_starts[r]), int(row_ends[r])
        for s in range(S):
            lo = dcp_layout.local_count(st, s, S, I)
            hi = dcp_layout.local_count(en, s, S, I)
            local_idx[s, j] = indexer.shard_topk(local_logits[s, r], lo, hi, K)
            sc, gid = indexer.pack(local_logits[s, r], local_idx[s, j], s, S, I)
            cand_sc[j, s * K:(s + 1) * K] = sc
            cand_id[j, s * K:(s + 1) * K] = gid
        ids[j], scores[j] = indexer.merge(cand_sc[j], cand_id[j], K)
    out = dict(rows=rows, local_idx=local_idx, cand_scores=cand_sc, cand_ids=cand_id,
               ids=ids, scores=scores)
    if tables is not None:
        slots = np.full((S, n, K), -1, np.int64)
        counts = np.zeros((S, n), np.int64)
        err = False
        for j, r in enumerate(rows):
            q = int(r if row_to_req is None else row_to_req[r])
            sl, cnt, e = indexer.convert_compact(ids[j], S, I, tables[:, q], block_size)
            slots[:, j], counts[:, j] = sl, cnt
            err |= e
        out.update(slots=slots, counts=counts, error=err)
    return out
