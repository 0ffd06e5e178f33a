"""LSE combine of per-shard partial attention outputs, in fp64.  Test infrastructure.

Sources: PR #46076 report, "[Attention][DSA] support dcp for
FLASHINFER_MLA_SPARSE", section 实现拆解 item 5 and section 评论区精华 "LSE base
normalisation": the sparse MLA kernel returns a base-2 LSE, the DCP reducer
expects base-e, so `_normalize_lse` converts first.  PR #52046 report, "DSV3.2
PCP sharding", section 关键源码片段: `dcp_manager.combine(attn_out, lse, ...)`
merges the shards' partial outputs by their LSE.  The merge formula is not
printed on the pages; the one below is the exact softmax identity it must
compute: with lambda_s = ln(sum of exp(score) over shard s's tokens) and O_s the
shard's softmax-weighted value average,

    O = sum_s exp(lambda_s) O_s / sum_s exp(lambda_s),   lse = ln sum_s exp(lambda_s).

Reading where the pages are silent: a shard that holds no selected token has
lse2 = -inf (its output is ignored); when every shard is empty the result is
O = 0 and lse = -inf.
"""
from __future__ import annotations

import numpy as np

LN2 = np.log(2.0)


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as fp64."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def lse_combine(partial, lse2):
    """partial [S, ..., D] fp64 values, lse2 [S, ...] base-2 LSE.

    Returns (out [..., D] fp64 unrounded, lse [...] fp64 base-e).
    """
    partial = np.asarray(partial, np.float64)
    lam = np.asarray(lse2, np.float64) * LN2           # base 2 -> base e
    M = lam.max(axis=0)
    empty = np.isneginf(M)
    Msafe = np.where(empty, 0.0, M)
    w = np.exp(lam - Msafe[None])                      # exp(-inf) = 0 for empty shards
    wsum = w.sum(axis=0)
    # An empty shard's output does not take part (0 * value would still be fine
    # for finite values; masking keeps the definition independent of them).
    contrib = np.where((w > 0)[..., None], w[..., None] * partial, 0.0)
    num = contrib.sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(empty[..., None], 0.0, num / np.where(empty, 1.0, wsum)[..., None])
        lse = np.where(empty, -np.inf, Msafe + np.log(np.where(empty, 1.0, wsum)))
    return out, lse
