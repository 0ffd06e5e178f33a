"""Interleaved DCP sharding of a token sequence, by definition.  Test infrastructure.

The rule (PR #46076 report "[Attention][DSA] support dcp for
FLASHINFER_MLA_SPARSE", section 关键源码片段 / key source snippets, the comment in
`_dcp_localize_decode_seq_lens`): a rank owns every token whose position `pos`
satisfies (pos // interleave) % dcp_world_size == rank.

Everything else here is derived from that rule by counting, never by a closed
form: a shard keeps the tokens it owns in increasing global order, so a token's
local slot is the number of tokens before it that the same shard owns, and a
shard's local length for a prefix [0, L) is the number of tokens in it that the
shard owns.  (The CUDA path uses closed forms instead; the tests check the two
agree.)
"""
from __future__ import annotations

import numpy as np


def owner(t, S: int, I: int):
    """Shard holding global token t: (t // I) mod S."""
    return (np.asarray(t, np.int64) // I) % S


def owned_tokens(L: int, s: int, S: int, I: int) -> np.ndarray:
    """Global ids in [0, L) that shard s holds, ascending (= its local order)."""
    t = np.arange(L, dtype=np.int64)
    return t[owner(t, S, I) == s]


def local_count(L: int, s: int, S: int, I: int) -> int:
    """Number of tokens of the prefix [0, L) that shard s holds."""
    return int(np.count_nonzero(owner(np.arange(L, dtype=np.int64), S, I) == s))


def local_counts(lengths, s: int, S: int, I: int) -> np.ndarray:
    """local_count for many prefix lengths at once (a running count)."""
    lengths = np.asarray(lengths, np.int64)
    top = int(lengths.max(initial=0))
    held = owner(np.arange(top, dtype=np.int64), S, I) == s
    running = np.concatenate([[0], np.cumsum(held)])
    return running[lengths].astype(np.int64)


def global_to_local(t, S: int, I: int):
    """(shard, local slot) of global token(s) t, by counting earlier tokens."""
    t = np.asarray(t, np.int64)
    top = int(t.max(initial=-1)) + 1
    own = owner(np.arange(top, dtype=np.int64), S, I)
    s = owner(t, S, I)
    slot = np.empty_like(t)
    for shard in np.unique(s):
        running = np.cumsum(own == shard) - 1          # slot of each held token
        sel = s == shard
        slot[sel] = running[t[sel]]
    return s, slot


def local_to_global(s: int, slots, S: int, I: int) -> np.ndarray:
    """Global id of local slot(s) of shard s: the slot-th token shard s holds."""
    slots = np.asarray(slots, np.int64)
    need = max(int(slots.max(initial=-1)) + 1, 1)
    # Every run of I*S consecutive tokens gives shard s exactly I of them, so the
    # first ceil(need / I) runs hold at least `need` of its tokens.
    toks = owned_tokens(-(-need // I) * I * S, s, S, I)
    return toks[slots]


def shard_rows(x: np.ndarray, row_ends, S: int, I: int, ld: int,
               fill: float | None = None) -> np.ndarray:
    """Split global logits rows x[rows, L] into the per-shard layout [S, rows, ld].

    out[s, r, l] is the value of the l-th token shard s holds.  This is what each
    DCP rank would see in its own memory; simulating S ranks on one device
    concatenates them along the leading axis.  Entries for tokens at or past a
    row's end are set to `fill` when given (a canary: the path must not read
    them); slots beyond the last held token keep `fill` too (0 when None).
    """
    rows, L = x.shape
    out = np.full((S, rows, ld), 0.0 if fill is None else fill, np.float32)
    row_ends = np.asarray(row_ends, np.int64)
    for s in range(S):
        toks = owned_tokens(L, s, S, I)
        n = min(len(toks), ld)
        vals = x[:, toks[:n]]
        if fill is not None:
            vals = np.where(toks[None, :n] < row_ends[:, None], vals, np.float32(fill))
        out[s, :, :n] = vals
    return out
