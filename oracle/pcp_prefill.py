"""The PCP prefill path's cache-row production: RMS norm of the latent kv_c,
rotary embedding of k_pe, the rows materialised for the gather, and their
insertion into the paged KV cache.  Test infrastructure; fp64.

Source (page title and sections): PR #52046 report, "DSV3.2 PCP sharding":
  功能与动机 (motivation): with PCP the sequence is sharded across ranks while
      the KV cache is replicated like TP, so the cache rows a forward produces
      must be gathered before they are inserted; fused_norm_rope therefore
      materialises its outputs instead of writing the cache directly.
  实现拆解 item 1 and 关键源码片段 (`_fused_norm_rope_kernel`, the pid == 1
      branch): kv_c is RMS-normed with its weight; k_pe is rotated in the
      interleaved layout, each adjacent pair (x1, x2) = (k_pe[2i], k_pe[2i+1])
      becoming (x1 cos - x2 sin, x2 cos + x1 sin); with output buffers the
      results are stored there, and with a slot mapping the cache row at the
      token's slot receives kv_c then the rotated k_pe at its tail.
  实现拆解 item 3 (`maybe_gather_mla_latent_cache_inputs`, `do_kv_cache_update`):
      the ranks' materialised rows are gathered, then inserted into the cache.

Readings where the page is silent (listed with the others in the design
notes): the RMS norm is x / sqrt(mean(x^2) + eps) * weight; the rotation's
cos and sin come from a per-position table (cos in its first half, sin in its
second, one angle per pair), as the kernel's `cos`/`sin` operands; a slot of
-1 writes nothing; the ranks hold contiguous slices of the sequence, rank p
the p-th, so the gather is their concatenation in rank order.
"""
from __future__ import annotations

import numpy as np


def rms_norm(x, weight, eps: float) -> np.ndarray:
    """x [T, d], weight [d] -> x / sqrt(mean(x^2) + eps) * weight (fp64)."""
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, np.float64)


def rope_interleaved(x, cos, sin) -> np.ndarray:
    """x [T, 2n]; cos, sin [T, n]: pair i = (x[2i], x[2i+1]) rotated by the
    angle whose cosine and sine are cos[:, i], sin[:, i]."""
    x = np.asarray(x, np.float64)
    x1, x2 = x[:, 0::2], x[:, 1::2]
    c, s = np.asarray(cos, np.float64), np.asarray(sin, np.float64)
    out = np.empty_like(x)
    out[:, 0::2] = x1 * c - x2 * s
    out[:, 1::2] = x2 * c + x1 * s
    return out


def fused_norm_rope(kv_c, k_pe, weight, eps: float, positions, cos_sin_cache):
    """One rank's new tokens: (normed kv_c [T, d_c], rotated k_pe [T, d_r]).

    kv_c [T, d_c], k_pe [T, d_r] fp64 values; positions [T] int;
    cos_sin_cache [max_pos, d_r] (cos of the d_r / 2 pair angles, then sin)."""
    cs = np.asarray(cos_sin_cache, np.float64)[np.asarray(positions, np.int64)]
    half = cs.shape[1] // 2
    return rms_norm(kv_c, weight, eps), rope_interleaved(k_pe, cs[:, :half], cs[:, half:])


def gather_ranks(slices) -> np.ndarray:
    """The ranks' materialised rows (rank p holding the p-th contiguous slice
    of the sequence) in token order: their concatenation."""
    return np.concatenate([np.asarray(s) for s in slices], axis=0)


def cache_insert(cache, rows, slot_mapping) -> np.ndarray:
    """A copy of cache [n_slots, d] with row t written at slot_mapping[t]
    (slots < 0 skipped)."""
    out = np.array(cache, copy=True)
    slots = np.asarray(slot_mapping, np.int64)
    keep = slots >= 0
    out[slots[keep]] = np.asarray(rows)[keep]
    return out
