"""Torch-facing binding of the C ABI: argument checks and marshalling only.

Every function here validates dtype / device / contiguity, passes raw device
pointers and the current CUDA stream to libdsa.so, and returns the output
tensors.  No step of the path is computed in Python and there is no CPU path:
CPU tensors are rejected.
"""
from __future__ import annotations

import torch

from . import _lib

__all__ = ["shard_topk", "pack_candidates", "shard_topk_pack", "merge_topk_stable",
           "convert_index_compact", "indexer_fused", "lse_combine", "slot_mapping",
           "sparse_mla_decode", "new_error_flags", "SUPPORTED_K", "MLA_DQK", "MLA_DV"]

SUPPORTED_K = (512, 1024, 2048)
MLA_DQK, MLA_DV = 576, 512       # DSA_MLA_DQK, DSA_MLA_DV of include/dsa.h


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, dim: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def new_error_flags(device) -> torch.Tensor:
    """A zeroed device word for the kernels' DSA_FLAG_* bits."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def shard_topk(logits, row_ends, K: int, I: int, row_starts=None, out=None, err_flags=None):
    """Local top-K of every shard.  logits [S, rows, ld] fp32 -> [S, rows, K] int32."""
    _need(logits, "logits", torch.float32, 3)
    S, rows, ld = logits.shape
    _need(row_ends, "row_ends", torch.int32, 1)
    if row_starts is not None:
        _need(row_starts, "row_starts", torch.int32, 1)
    if out is None:
        out = torch.empty((S, rows, K), dtype=torch.int32, device=logits.device)
    _need(out, "out", torch.int32, 3)
    _lib.call("dsa_shard_topk", _ptr(logits), ld, rows, S, I, K, _ptr(row_starts),
              _ptr(row_ends), _ptr(out), _ptr(err_flags), _stream(logits))
    return out


def pack_candidates(logits, local_idx, I: int, out=None, err_flags=None):
    """(score, global id) candidates: -> [rows, S*K, 2] fp32 (id lane = int32 bits)."""
    _need(logits, "logits", torch.float32, 3)
    _need(local_idx, "local_idx", torch.int32, 3)
    S, rows, ld = logits.shape
    K = local_idx.shape[2]
    if out is None:
        out = torch.empty((rows, S * K, 2), dtype=torch.float32, device=logits.device)
    _need(out, "out", torch.float32, 3)
    _lib.call("dsa_pack_candidates", _ptr(logits), ld, _ptr(local_idx), rows, S, I, K,
              _ptr(out), _ptr(err_flags), _stream(logits))
    return out


def shard_topk_pack(logits, row_ends, K: int, I: int, row_starts=None, local_idx=None,
                    cand=None, want_local_idx: bool = True, err_flags=None):
    """Fused shard top-K + pack.  Returns (local_idx or None, cand)."""
    _need(logits, "logits", torch.float32, 3)
    S, rows, ld = logits.shape
    _need(row_ends, "row_ends", torch.int32, 1)
    if row_starts is not None:
        _need(row_starts, "row_starts", torch.int32, 1)
    if local_idx is None and want_local_idx:
        local_idx = torch.empty((S, rows, K), dtype=torch.int32, device=logits.device)
    if cand is None:
        cand = torch.empty((rows, S * K, 2), dtype=torch.float32, device=logits.device)
    _need(cand, "cand", torch.float32, 3)
    if local_idx is not None:
        _need(local_idx, "local_idx", torch.int32, 3)
    _lib.call("dsa_shard_topk_pack", _ptr(logits), ld, rows, S, I, K, _ptr(row_starts),
              _ptr(row_ends), _ptr(local_idx), _ptr(cand), _ptr(err_flags), _stream(logits))
    return local_idx, cand


def merge_topk_stable(cand, K: int, ids=None, scores=None, want_scores: bool = False,
                      err_flags=None):
    """Stable global top-K of [rows, C, 2] candidates -> ids [rows, K] (, scores)."""
    _need(cand, "cand", torch.float32, 3)
    rows, C, _two = cand.shape
    if ids is None:
        ids = torch.empty((rows, K), dtype=torch.int32, device=cand.device)
    _need(ids, "ids", torch.int32, 2)
    if scores is None and want_scores:
        scores = torch.empty((rows, K), dtype=torch.float32, device=cand.device)
    if scores is not None:
        _need(scores, "scores", torch.float32, 2)
    _lib.call("dsa_merge_topk_stable", _ptr(cand), rows, C, K, _ptr(ids), _ptr(scores),
              _ptr(err_flags), _stream(cand))
    return (ids, scores) if (want_scores or scores is not None) else ids


def convert_index_compact(ids, block_table, block_size: int, I: int, row_to_req=None,
                          slots=None, counts=None, want_counts: bool = True, err_flags=None):
    """Merged ids [rows, K] -> per-shard slots [S, rows, K] (, counts [S, rows])."""
    _need(ids, "ids", torch.int32, 2)
    _need(block_table, "block_table", torch.int32, 3)
    rows, K = ids.shape
    S, reqs, max_blocks = block_table.shape
    if row_to_req is not None:
        _need(row_to_req, "row_to_req", torch.int32, 1)
    if slots is None:
        slots = torch.empty((S, rows, K), dtype=torch.int32, device=ids.device)
    _need(slots, "slots", torch.int32, 3)
    if counts is None and want_counts:
        counts = torch.empty((S, rows), dtype=torch.int32, device=ids.device)
    if counts is not None:
        _need(counts, "counts", torch.int32, 2)
    _lib.call("dsa_convert_index_compact", _ptr(ids), rows, K, S, I, _ptr(block_table), reqs,
              max_blocks, block_size, _ptr(row_to_req), _ptr(slots), _ptr(counts),
              _ptr(err_flags), _stream(ids))
    return slots, counts


def indexer_fused(logits, row_ends, K: int, I: int, block_table, block_size: int,
                  row_starts=None, row_to_req=None, ids=None, slots=None, counts=None,
                  want_scores: bool = False, want_local_idx: bool = False,
                  want_cand: bool = False, err_flags=None, scores=None, local_idx=None,
                  cand=None) -> dict:
    """Shard top-K, pack, merge and convert in one kernel (S <= 8).

    Returns a dict with ids [rows, K], slots [S, rows, K], counts [S, rows] and,
    when asked for (or given as output tensors), scores, local_idx and cand."""
    _need(logits, "logits", torch.float32, 3)
    S, rows, ld = logits.shape
    _need(row_ends, "row_ends", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 3)
    if block_table.shape[0] != S:
        raise ValueError("block_table must be [S, reqs, max_blocks]")
    _, reqs, max_blocks = block_table.shape
    for name, t in (("row_starts", row_starts), ("row_to_req", row_to_req)):
        if t is not None:
            _need(t, name, torch.int32, 1)
    dv = logits.device
    out = {
        "ids": ids if ids is not None else torch.empty((rows, K), dtype=torch.int32, device=dv),
        "slots": slots if slots is not None else
        torch.empty((S, rows, K), dtype=torch.int32, device=dv),
        "counts": counts if counts is not None else
        torch.empty((S, rows), dtype=torch.int32, device=dv),
        "scores": scores if scores is not None else
        torch.empty((rows, K), dtype=torch.float32, device=dv) if want_scores else None,
        "local_idx": local_idx if local_idx is not None else
        torch.empty((S, rows, K), dtype=torch.int32, device=dv) if want_local_idx else None,
        "cand": cand if cand is not None else
        torch.empty((rows, S * K, 2), dtype=torch.float32, device=dv) if want_cand else None,
    }
    for name, dt, nd in (("scores", torch.float32, 2), ("local_idx", torch.int32, 3),
                         ("cand", torch.float32, 3)):
        if out[name] is not None:
            _need(out[name], name, dt, nd)
    _need(out["ids"], "ids", torch.int32, 2)
    _need(out["slots"], "slots", torch.int32, 3)
    _need(out["counts"], "counts", torch.int32, 2)
    _lib.call("dsa_indexer_fused", _ptr(logits), ld, rows, S, I, K, _ptr(row_starts),
              _ptr(row_ends), _ptr(block_table), reqs, max_blocks, block_size, _ptr(row_to_req),
              _ptr(out["ids"]), _ptr(out["scores"]), _ptr(out["slots"]), _ptr(out["counts"]),
              _ptr(out["local_idx"]), _ptr(out["cand"]), _ptr(err_flags), _stream(logits))
    return out


def lse_combine(partial_out, lse2, out=None, lse_out=None, want_lse: bool = True,
                err_flags=None):
    """partial_out [S, rows, H, D] bf16, lse2 [S, rows, H] fp32 (base 2)
    -> out [rows, H, D] bf16 (, lse [rows, H] fp32 base e)."""
    _need(partial_out, "partial_out", torch.bfloat16, 4)
    _need(lse2, "lse2", torch.float32, 3)
    S, rows, H, D = partial_out.shape
    if tuple(lse2.shape) != (S, rows, H):
        raise ValueError("lse2 must be [S, rows, H]")
    if out is None:
        out = torch.empty((rows, H, D), dtype=torch.bfloat16, device=partial_out.device)
    _need(out, "out", torch.bfloat16, 3)
    if lse_out is None and want_lse:
        lse_out = torch.empty((rows, H), dtype=torch.float32, device=partial_out.device)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, 2)
    _lib.call("dsa_lse_combine", _ptr(partial_out), _ptr(lse2), S, rows, H, D, _ptr(out),
              _ptr(lse_out), _ptr(err_flags), _stream(partial_out))
    return out, lse_out


def slot_mapping(positions, block_table, block_size: int, I: int, token_req=None, out=None,
                 err_flags=None):
    """Write-side KV slots of new tokens: positions [n] int32 (and token_req [n],
    default token i = request i) -> [S, n] int32, -1 where a shard does not
    store the token."""
    _need(positions, "positions", torch.int32, 1)
    _need(block_table, "block_table", torch.int32, 3)
    S, reqs, max_blocks = block_table.shape
    n = positions.shape[0]
    if token_req is not None:
        _need(token_req, "token_req", torch.int32, 1)
        if token_req.shape[0] != n:
            raise ValueError("token_req must have one entry per position")
    if out is None:
        out = torch.empty((S, n), dtype=torch.int32, device=positions.device)
    _need(out, "out", torch.int32, 2)
    _lib.call("dsa_slot_mapping", _ptr(positions), _ptr(token_req), n, S, I, _ptr(block_table),
              reqs, max_blocks, block_size, _ptr(out), _ptr(err_flags), _stream(positions))
    return out


def sparse_mla_decode(q, kv_cache, slots, counts, scale: float, out=None, lse2=None,
                      err_flags=None):
    """Each shard's sparse MLA decode attention over its compacted slots.

    q [rows, H, 576] bf16, kv_cache [S, n_slots, 576] bf16, slots [S, rows, K]
    int32, counts [S, rows] int32 -> (out [S, rows, H, 512] bf16, lse2 [S, rows, H]
    fp32, base 2)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", torch.bfloat16, 3)
    _need(slots, "slots", torch.int32, 3)
    _need(counts, "counts", torch.int32, 2)
    rows, H, dqk = q.shape
    S, n_slots, dqk2 = kv_cache.shape
    if dqk != MLA_DQK or dqk2 != MLA_DQK:
        raise ValueError(f"q and kv_cache rows must have {MLA_DQK} entries")
    if slots.shape[:2] != (S, rows) or tuple(counts.shape) != (S, rows):
        raise ValueError("slots must be [S, rows, K] and counts [S, rows]")
    K = slots.shape[2]
    if out is None:
        out = torch.empty((S, rows, H, MLA_DV), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    if lse2 is None:
        lse2 = torch.empty((S, rows, H), dtype=torch.float32, device=q.device)
    _need(lse2, "lse2", torch.float32, 3)
    _lib.call("dsa_sparse_mla_decode", _ptr(q), _ptr(kv_cache), n_slots, _ptr(slots),
              _ptr(counts), rows, S, H, K, float(scale), _ptr(out), _ptr(lse2), _ptr(err_flags),
              _stream(q))
    return out, lse2


IDX_HEADS, IDX_DIM = 64, 128


def indexer_logits(q, weights, k_cache, block_table, block_size: int, row_ends, I: int,
                   ld: int, row_starts=None, row_to_req=None, out=None, err_flags=None):
    """Each shard's indexer logits over its local slots.

    q [rows, 64, 128] uint8 (fp8 e4m3 codes), weights [rows, 64] fp32,
    k_cache [S, n_slots, 128] uint8 (e4m3), block_table [S, reqs, max_blocks]
    -> logits [S, rows, ld] fp32 (only each row's local range is written)."""
    _need(q, "q", torch.uint8, 3)
    _need(weights, "weights", torch.float32, 2)
    _need(k_cache, "k_cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 3)
    _need(row_ends, "row_ends", torch.int32, 1)
    rows = q.shape[0]
    if tuple(q.shape[1:]) != (IDX_HEADS, IDX_DIM) or tuple(weights.shape) != (rows, IDX_HEADS):
        raise ValueError("q must be [rows, 64, 128] and weights [rows, 64]")
    S, n_slots, dim = k_cache.shape
    if dim != IDX_DIM or block_table.shape[0] != S:
        raise ValueError("k_cache must be [S, n_slots, 128] and block_table [S, reqs, max_blocks]")
    _, reqs, max_blocks = block_table.shape
    for name, t in (("row_starts", row_starts), ("row_to_req", row_to_req)):
        if t is not None:
            _need(t, name, torch.int32, 1)
    if out is None:
        out = torch.empty((S, rows, ld), dtype=torch.float32, device=q.device)
    _need(out, "out", torch.float32, 3)
    if tuple(out.shape) != (S, rows, ld):
        raise ValueError("out must be [S, rows, ld]")
    _lib.call("dsa_indexer_logits", _ptr(q), _ptr(weights), _ptr(k_cache), n_slots,
              _ptr(block_table), reqs, max_blocks, block_size, _ptr(row_to_req),
              _ptr(row_starts), _ptr(row_ends), rows, S, I, _ptr(out), ld, _ptr(err_flags),
              _stream(q))
    return out


def fused_norm_rope(kv_c, k_pe, positions, norm_weight, eps: float, cos_sin_cache,
                    materialize: bool = True, slot_mapping=None, kv_cache=None, kv_out=None,
                    kpe_out=None, err_flags=None):
    """New tokens' cache rows: kv_c [T, 512] bf16 RMS-normed, k_pe [T, 64] bf16
    rotated (interleaved pairs) by cos_sin_cache [max_pos, 64] fp32 at
    positions [T].  Returns (kv_out, kpe_out) when materialising (else
    (None, None)); with slot_mapping [T] and kv_cache [n_slots, 576] bf16, row
    slot_mapping[t] of the cache is written as well."""
    _need(kv_c, "kv_c", torch.bfloat16, 2)
    _need(k_pe, "k_pe", torch.bfloat16, 2)
    _need(positions, "positions", torch.int32, 1)
    _need(norm_weight, "norm_weight", torch.float32, 1)
    _need(cos_sin_cache, "cos_sin_cache", torch.float32, 2)
    T = kv_c.shape[0]
    if tuple(kv_c.shape) != (T, MLA_DV) or tuple(k_pe.shape) != (T, MLA_DQK - MLA_DV):
        raise ValueError("kv_c must be [T, 512] and k_pe [T, 64]")
    if cos_sin_cache.shape[1] != MLA_DQK - MLA_DV:
        raise ValueError("cos_sin_cache must be [max_pos, 64]")
    if materialize:
        if kv_out is None:
            kv_out = torch.empty((T, MLA_DV), dtype=torch.bfloat16, device=kv_c.device)
        if kpe_out is None:
            kpe_out = torch.empty((T, MLA_DQK - MLA_DV), dtype=torch.bfloat16, device=kv_c.device)
        _need(kv_out, "kv_out", torch.bfloat16, 2)
        _need(kpe_out, "kpe_out", torch.bfloat16, 2)
    else:
        kv_out = kpe_out = None
    n_slots = 0
    if slot_mapping is not None or kv_cache is not None:
        _need(slot_mapping, "slot_mapping", torch.int32, 1)
        _need(kv_cache, "kv_cache", torch.bfloat16, 2)
        n_slots = kv_cache.shape[0]
    _lib.call("dsa_fused_norm_rope", _ptr(kv_c), _ptr(k_pe), _ptr(positions), _ptr(norm_weight),
              float(eps), _ptr(cos_sin_cache), cos_sin_cache.shape[0], T, _ptr(kv_out),
              _ptr(kpe_out), _ptr(slot_mapping), _ptr(kv_cache), n_slots, _ptr(err_flags),
              _stream(kv_c))
    return kv_out, kpe_out


def kv_cache_insert(kv_rows, kpe_rows, slot_mapping, kv_cache, err_flags=None):
    """Gathered rows (kv_rows [T, 512], kpe_rows [T, 64] bf16) into
    kv_cache [n_slots, 576] bf16 at slot_mapping [T] (-1: skipped)."""
    _need(kv_rows, "kv_rows", torch.bfloat16, 2)
    _need(kpe_rows, "kpe_rows", torch.bfloat16, 2)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    _need(kv_cache, "kv_cache", torch.bfloat16, 2)
    T = kv_rows.shape[0]
    _lib.call("dsa_kv_cache_insert", _ptr(kv_rows), _ptr(kpe_rows), _ptr(slot_mapping), T,
              _ptr(kv_cache), kv_cache.shape[0], _ptr(err_flags), _stream(kv_rows))
    return kv_cache
