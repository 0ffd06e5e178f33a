"""Seeded synthetic inputs for the DCP sparse-indexer path.

This module is the only code shared by the CPU oracle and the CUDA path.  It
holds random draws and data-format helpers only: no step of the method (no
ownership rule, no top-K, no slot mapping, no LSE arithmetic).  Anything that
depends on how tokens are split across shards is passed in by the caller.

Every workload below follows one of the five shapes the DeepSeek-V3.2 / GLM
sparse-indexer DCP pages describe (PR #46076 report "[Attention][DSA] support
dcp for FLASHINFER_MLA_SPARSE": DCP decode with index_topk in 512/1024/2048;
PR #52046 report "DSV3.2 PCP sharding": 32k-token prefill chunks).  No public
dataset or model weights are involved; the numbers are synthetic stand-ins.

Sizes that follow from the sharding (the per-shard row stride `ld` and the
block-table width `max_blocks`) are listed as plain numbers in CONFIGS; how
they were derived is written next to each entry.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "Config", "CONFIGS", "rng_for", "row_ranges", "global_logits",
    "iid_local_logits", "block_tables", "combine_inputs",
    "f32_to_bf16_bits", "IDX_HEADS", "IDX_DIM", "e4m3_codes", "indexer_query",
    "indexer_weights", "indexer_keys", "PCP_DC", "PCP_DR", "pcp_token_inputs",
    "rotation_table",
]


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    index: int          # position in the workload list; seeds derive from it
    rows: int           # query rows (decode tokens or prefill rows)
    S: int              # logical shards (DCP world size)
    I: int              # interleave size
    K: int              # index_topk
    block_size: int
    max_len: int        # longest global row
    ld: int             # per-shard logits row stride (>= longest local row, multiple of 4)
    reqs: int           # rows of each shard's block table
    max_blocks: int     # block-table columns
    H: int = 0          # combine heads (0: no combine inputs in the recipe)
    D: int = 0          # combine head dim
    description: str = ""


# ld and max_blocks: the longest local row of a shard is the token count shard 0
# owns in [0, max_len); for these sizes that is max_len / S (all max_len are
# multiples of I*S).  max_blocks = ceil(ld / block_size).
CONFIGS = {
    "tiny": Config(
        "tiny", 0, rows=4, S=2, I=1, K=512, block_size=64, max_len=4096,
        ld=2048, reqs=4, max_blocks=32,
        description="4 rows, seq 4096, S=2, I=1, K=512; logits on a 1/64 grid "
                    "(forces ties and -0.0); identity block table"),
    "decode": Config(
        "decode", 1, rows=64, S=4, I=1, K=2048, block_size=64, max_len=65536,
        ld=16384, reqs=64, max_blocks=256, H=128, D=512,
        description="64 decode rows, S=4, I=1, K=2048, seq_len ~ U[8192, 65536], "
                    "N(0,1) logits, per-shard randomly permuted paged blocks"),
    "long_decode": Config(
        "long_decode", 2, rows=128, S=8, I=16, K=2048, block_size=64,
        max_len=131072, ld=16384, reqs=128, max_blocks=256,
        description="128 rows, S=8, I=16, K=2048, seq 131072; 10% of logits "
                    "duplicate an earlier token's value (heavy ties)"),
    "prefill": Config(
        "prefill", 3, rows=4096, S=4, I=1, K=2048, block_size=64, max_len=32768,
        ld=8192, reqs=1, max_blocks=128,
        description="4096 causal rows over a 32768-token context, row i sees "
                    "[0, 28672+i); S=4, I=1, K=2048; -inf beyond the row end"),
    "ragged": Config(
        "ragged", 4, rows=256, S=8, I=4, K=1024, block_size=64, max_len=65536,
        ld=8192, reqs=256, max_blocks=128, H=128, D=512,
        description="256 rows, S=8, I=4, K=1024, seq_len log-uniform in "
                    "[16, 65536] (rows shorter than K and than I*S); combine of "
                    "[256,128,512] bf16 partial outputs with base-2 LSE in [-5, 20]"),
}

# Sub-seeds: one per buffer so that buffers can be drawn independently.
_SUB = {"lens": 1, "logits": 2, "dup_mask": 3, "dup_src": 4, "tables": 5,
        "out": 6, "lse": 7}


def rng_for(cfg: Config, buffer: str, replica: int = 0) -> np.random.Generator:
    """PCG64 stream for one buffer of one workload (seed = index*1000 + 17)."""
    return np.random.default_rng([cfg.index * 1000 + 17, _SUB[buffer], replica])


def row_ranges(cfg: Config, replica: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Global [row_start, row_end) of every row, int32 (row_start is 0 throughout)."""
    rows = cfg.rows
    starts = np.zeros(rows, np.int32)
    if cfg.name in ("tiny", "long_decode"):
        ends = np.full(rows, cfg.max_len, np.int32)
    elif cfg.name == "decode":
        ends = rng_for(cfg, "lens", replica).integers(
            8192, 65536, size=rows, endpoint=True).astype(np.int32)
    elif cfg.name == "prefill":
        ends = (28672 + np.arange(rows)).astype(np.int32)
    elif cfg.name == "ragged":
        u = rng_for(cfg, "lens", replica).uniform(math.log(16), math.log(65536), rows)
        ends = np.floor(np.exp(u)).astype(np.int32)
        ends = np.clip(ends, 16, 65536)
    else:
        raise KeyError(cfg.name)
    return starts, ends


def global_logits(cfg: Config, replica: int = 0) -> np.ndarray:
    """fp32 indexer logits in global token order, shape [rows, max_len].

    Entries at or beyond a row's end are never read by the path; the prefill
    recipe fills them with -inf (the causal mask), the others leave N(0,1).
    """
    rows, L = cfg.rows, cfg.max_len
    rng = rng_for(cfg, "logits", replica)
    x = rng.standard_normal((rows, L), dtype=np.float32)
    if cfg.name == "tiny":
        x = (np.rint(x * np.float32(64.0)) / np.float32(64.0)).astype(np.float32)
    elif cfg.name == "long_decode":
        x = _with_duplicates(x, rng_for(cfg, "dup_mask", replica),
                             rng_for(cfg, "dup_src", replica), p=0.1)
    elif cfg.name == "prefill":
        _, ends = row_ranges(cfg, replica)
        cols = np.arange(L)[None, :]
        x[cols >= ends[:, None]] = -np.inf
    return x


def _with_duplicates(base: np.ndarray, rng_mask, rng_src, p: float) -> np.ndarray:
    """For t > 0, with probability p token t copies the value of a uniformly
    drawn earlier token u in [0, t); otherwise it keeps its own N(0,1) draw."""
    rows, L = base.shape
    t = np.arange(L)
    dup = rng_mask.random((rows, L)) < p
    dup[:, 0] = False
    u = np.floor(rng_src.random((rows, L)) * t[None, :]).astype(np.int64)
    src = np.where(dup, u, t[None, :])
    # Copies may chain (u itself a copy); resolve by pointer jumping (u < t).
    while True:
        nxt = np.take_along_axis(src, src, axis=1)
        if np.array_equal(nxt, src):
            break
        src = nxt
    return np.take_along_axis(base, src, axis=1)


def iid_local_logits(cfg: Config, replica: int = 0) -> np.ndarray:
    """[S, rows, ld] fp32 i.i.d. N(0,1): a per-shard layout drawn directly.

    For the N(0,1) recipes the values are independent of the token, so drawing
    each shard's local rows directly has the same distribution as splitting a
    global row; no ownership rule is needed.  Used where the workload needs no
    cross-token structure (ties, masks) and the oracle is not consulted.
    """
    rng = rng_for(cfg, "logits", replica)
    return rng.standard_normal((cfg.S, cfg.rows, cfg.ld), dtype=np.float32)


def block_tables(cfg: Config, identity: bool | None = None, replica: int = 0) -> np.ndarray:
    """[S, reqs, max_blocks] int32 paged block tables.

    Identity (tiny recipe): request q's column c maps to block q*max_blocks + c.
    Otherwise each shard's physical blocks are an independent random
    permutation of [0, reqs*max_blocks) laid out row-major.
    """
    S, R, B = cfg.S, cfg.reqs, cfg.max_blocks
    if identity is None:
        identity = cfg.name == "tiny"
    if identity:
        one = np.arange(R * B, dtype=np.int32).reshape(R, B)
        return np.broadcast_to(one, (S, R, B)).copy()
    rng = rng_for(cfg, "tables", replica)
    return np.stack([rng.permutation(R * B).astype(np.int32).reshape(R, B)
                     for _ in range(S)])


def combine_inputs(cfg: Config, empty: np.ndarray | None = None, replica: int = 0,
                   rows: int | None = None):
    """Per-shard partial attention outputs and their base-2 LSE.

    Returns (out_bits uint16 [S, rows, H, D] as bf16 bit patterns,
    lse2 float32 [S, rows, H]).  Values are N(0,1) rounded to bf16 and
    lse2 ~ U[-5, 20].  `empty` [S, rows] bool marks (shard, row) pairs that
    hold no selected token: there lse2 = -inf and the output is zero.
    """
    S, H, D = cfg.S, cfg.H, cfg.D
    rows = cfg.rows if rows is None else rows
    rng_o = rng_for(cfg, "out", replica)
    rng_l = rng_for(cfg, "lse", replica)
    out = f32_to_bf16_bits(rng_o.standard_normal((S, rows, H, D), dtype=np.float32))
    lse2 = rng_l.uniform(-5.0, 20.0, (S, rows, H)).astype(np.float32)
    if empty is not None:
        empty = np.asarray(empty, bool)
        lse2[empty] = -np.inf
        out[empty] = 0
    return out, lse2


MLA_DQK, MLA_DV = 576, 512     # a cache row / query head: latent 512 + rope 64


def mla_query(rows: int, H: int, seed: int) -> np.ndarray:
    """[rows, H, 576] MQA queries (latent + rope parts), N(0,1) in bf16 bits."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((rows, H, MLA_DQK), dtype=np.float32))


def mla_cache(S: int, n_slots: int, seed: int) -> np.ndarray:
    """[S, n_slots, 576] paged KV caches by slot, N(0,1) in bf16 bits."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((S, n_slots, MLA_DQK), dtype=np.float32))


def mla_cache_uniform(S: int, n_slots: int, seed: int) -> np.ndarray:
    """[S, n_slots, 576] paged KV caches for benchmark-sized runs (gigabytes):
    bf16 bit patterns with a random sign, exponent -1 and 7 random mantissa
    bits, i.e. values of magnitude in [0.5, 1), drawn 16 bits at a time so that
    several gigabytes take seconds to draw."""
    rng = np.random.default_rng(seed)
    w = rng.integers(0, 1 << 16, (S, n_slots, MLA_DQK), dtype=np.uint16)
    w &= np.uint16(0x807F)
    w |= np.uint16(0x3F00)
    return w


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits.
    Inputs are finite."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    # finite inputs: the largest sum, 0xFF7FFFFF + 0x8000, still fits in uint32
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)



# Indexer-logits inputs: H_I = 64 query heads of d_I = 128 fp8 (e4m3) values per
# query token, one fp32 weight per head, one 128-value fp8 key per cached token.
IDX_HEADS, IDX_DIM = 64, 128


def e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Random fp8 e4m3 codes (uint8): a random sign, an exponent field drawn
    uniformly from 4..9 and three random mantissa bits, i.e. magnitudes in
    [2^-3, 2^2 * 1.875], roughly log-uniform; no NaN code, no subnormal."""
    sign = rng.integers(0, 2, shape, dtype=np.uint8) << np.uint8(7)
    expo = rng.integers(4, 10, shape, dtype=np.uint8) << np.uint8(3)
    mant = rng.integers(0, 8, shape, dtype=np.uint8)
    return sign | expo | mant


def indexer_query(rows: int, seed: int) -> np.ndarray:
    """[rows, 64, 128] fp8 e4m3 codes: the query heads of each query token."""
    return e4m3_codes(np.random.default_rng(seed), (rows, IDX_HEADS, IDX_DIM))


def indexer_weights(rows: int, seed: int) -> np.ndarray:
    """[rows, 64] fp32 head weights, N(0, 1/64)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((rows, IDX_HEADS), dtype=np.float32) / np.float32(8.0))


def indexer_keys(S: int, n_slots: int, seed: int) -> np.ndarray:
    """[S, n_slots, 128] fp8 e4m3 codes: each shard's paged indexer key cache
    by physical slot."""
    return e4m3_codes(np.random.default_rng(seed), (S, n_slots, IDX_DIM))


# PCP prefill inputs: each new token's latent kv_c (512) and rope part k_pe
# (64), bf16, the RMS-norm weight, and a per-position rotation table.
PCP_DC, PCP_DR = 512, 64


def pcp_token_inputs(T: int, seed: int):
    """(kv_c bits uint16 [T, 512], k_pe bits uint16 [T, 64], weight fp32 [512]):
    N(0,1) values rounded to bf16; weights 1 + N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    kv = f32_to_bf16_bits(rng.standard_normal((T, PCP_DC), dtype=np.float32))
    kpe = f32_to_bf16_bits(rng.standard_normal((T, PCP_DR), dtype=np.float32))
    w = (1.0 + 0.1 * rng.standard_normal(PCP_DC)).astype(np.float32)
    return kv, kpe, w


def rotation_table(max_pos: int, seed: int) -> np.ndarray:
    """[max_pos, 64] fp32 rotation table: for every position, the cosines then
    the sines of 32 angles drawn uniformly from [-pi, pi) (any angles serve:
    the path applies the table it is given)."""
    rng = np.random.default_rng(seed)
    ang = rng.uniform(-np.pi, np.pi, (max_pos, PCP_DR // 2))
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
