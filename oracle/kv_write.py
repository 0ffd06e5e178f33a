"""Write-side slot mapping of new tokens under DCP, by definition.  Test
infrastructure.

Sources (page titles and sections):
  [P40996] PR #40996 report, "DCP supports hybrid attention": section 实现拆解
           (implementation breakdown) item 2 (BlockTable and slot mapping: a
           token -> KV-slot mapping computed per rank, the allocation block
           may hold several kernel blocks, KV_CACHE_BLOCK_SIZE and
           BLOCKS_PER_KV_BLOCK) and item 1 (an attention group's rank keeps
           only its share of each sequence, in rank-local block tables).
  [P46076] PR #46076 report, "[Attention][DSA] support dcp for
           FLASHINFER_MLA_SPARSE": section 关键源码片段 (key source snippets),
           the ownership rule in `_dcp_localize_decode_seq_lens`.

Readings taken where the pages are silent (listed with the rest in the design
notes):
  * a rank stores a new token exactly when it owns it, at the token's local
    slot l (the number of earlier tokens of the same request the rank owns),
    through its own block table: entry tables[s, req, l // block_size], offset
    l % block_size; every other rank's mapping for that token is -1, which a
    cache insert skips;
  * block_size is the allocation block (KV_CACHE_BLOCK_SIZE); naming a kernel
    block of block_size / m tokens inside it (BLOCKS_PER_KV_BLOCK = m) changes
    the block numbering, not the slot;
  * a negative position is a padding token: -1 everywhere, not an error;
  * a request outside the table, a column past its width, a negative table
    entry or a slot past the int32 range of the output is an error: -1 for
    that token.
"""
from __future__ import annotations

import numpy as np

from . import dcp_layout


def slot_mapping(positions, token_req, S: int, I: int, tables, block_size: int):
    """Slots of new tokens on every shard [P40996 item 2; P46076 ownership rule].

    positions  [n] global positions of the new tokens in their requests
    token_req  [n] request of each token
    tables     [S, reqs, max_blocks] each shard's block table

    Returns (slots int64[S, n], error bool): slots[s, i] is token i's physical
    KV slot in shard s's cache when s owns it, else -1.
    """
    positions = np.asarray(positions, np.int64)
    token_req = np.asarray(token_req, np.int64)
    tables = np.asarray(tables, np.int64)
    reqs, max_blocks = tables.shape[1], tables.shape[2]
    n = positions.shape[0]
    out = np.full((S, n), -1, np.int64)
    error = False
    real = positions >= 0                      # negative positions: padding tokens
    shard = np.full(n, -1, np.int64)
    local = np.full(n, -1, np.int64)
    if real.any():
        shard[real], local[real] = dcp_layout.global_to_local(positions[real], S, I)
    for i in range(n):
        if not real[i]:
            continue
        s, l = int(shard[i]), int(local[i])
        req = int(token_req[i])
        col = l // block_size
        if not (0 <= req < reqs) or col >= max_blocks:
            error = True
            continue
        block = int(tables[s, req, col])
        if block < 0:
            error = True
            continue
        slot = block * block_size + l % block_size
        if slot > np.iinfo(np.int32).max:
            error = True
            continue
        out[s, i] = slot
    return out, error
