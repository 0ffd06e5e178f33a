"""Shared helpers for the GPU parity tests: build a workload's inputs, run the
CUDA path through the binding, run the oracle on sampled rows, compare."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import combine as OC
from oracle import dcp_layout as OL
from oracle import indexer as OX
from oracle import pipeline as OP


def row_to_req_for(cfg) -> np.ndarray | None:
    if cfg.reqs == cfg.rows:
        return None
    return np.zeros(cfg.rows, np.int32)          # prefill: every row is one request


def make_case(name: str, fill=None, replica: int = 0) -> dict:
    cfg = W.CONFIGS[name]
    starts, ends = W.row_ranges(cfg, replica)
    x = W.global_logits(cfg, replica)
    local = OL.shard_rows(x, ends, cfg.S, cfg.I, cfg.ld, fill=fill)
    return dict(cfg=cfg, x=x, local=local, starts=starts, ends=ends,
                bt=W.block_tables(cfg, replica=replica), r2q=row_to_req_for(cfg))


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


GUARD_BYTES = 4096
POISON = 0xA5


class Guards:
    """Output buffers with a poisoned 4 KB guard before and after each: a
    kernel that writes past either end of an output changes a guard byte.
    (Memory checkers are not available on the GPU hosts; these guards stand in
    for them on every output of the parity tests.)"""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype) -> torch.Tensor:
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((2 * GUARD_BYTES + n,), POISON, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n))
        return raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)

    def check(self) -> None:
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.bufs):
            head, tail = raw[:GUARD_BYTES], raw[GUARD_BYTES + n:]
            assert bool((head == POISON).all()), f"write before output buffer {i}"
            assert bool((tail == POISON).all()), f"write past output buffer {i}"


def run_gpu(case: dict, fused: bool = True) -> dict:
    """The launch sequence the benchmark times: fused shard top-K + pack, merge,
    convert, every output guarded.  Also returns the error word."""
    import dsa_sparse_indexer_gb300 as dsa
    cfg = case["cfg"]
    S, R, K = cfg.S, cfg.rows, cfg.K
    logits = dev(case["local"])
    starts = dev(case["starts"])
    ends = dev(case["ends"])
    bt = dev(case["bt"])
    r2q = None if case["r2q"] is None else dev(case["r2q"])
    err = dsa.new_error_flags("cuda")
    g = Guards()
    local_idx = g.empty((S, R, K), torch.int32)
    cand = g.empty((R, S * K, 2), torch.float32)
    if fused:
        dsa.shard_topk_pack(logits, ends, K, cfg.I, row_starts=starts, local_idx=local_idx,
                            cand=cand, err_flags=err)
        pack_err = err.clone()
        # The benchmark's call (no local indices) gives the same candidates
        # bit for bit.
        lean_err = dsa.new_error_flags("cuda")
        lean = g.empty((R, S * K, 2), torch.float32)
        dsa.shard_topk_pack(logits, ends, K, cfg.I, row_starts=starts, want_local_idx=False,
                            cand=lean, err_flags=lean_err)
        assert torch.equal(lean.view(torch.int32), cand.view(torch.int32)), "lean pack differs"
    else:
        dsa.shard_topk(logits, ends, K, cfg.I, row_starts=starts, out=local_idx, err_flags=err)
        dsa.pack_candidates(logits, local_idx, cfg.I, out=cand, err_flags=err)
    ids, scores = dsa.merge_topk_stable(cand, K, ids=g.empty((R, K), torch.int32),
                                        scores=g.empty((R, K), torch.float32), err_flags=err)
    slots, counts = dsa.convert_index_compact(ids, bt, cfg.block_size, cfg.I, row_to_req=r2q,
                                              slots=g.empty((S, R, K), torch.int32),
                                              counts=g.empty((S, R), torch.int32), err_flags=err)
    g.check()
    if fused:
        assert int(lean_err.item()) == int(pack_err.item()), "lean pack error word"
    cand_np = cand.cpu().numpy()
    return dict(local_idx=local_idx.cpu().numpy(), cand_scores=cand_np[..., 0],
                cand_ids=cand_np[..., 1].view(np.int32), ids=ids.cpu().numpy(),
                scores=scores.cpu().numpy(), slots=slots.cpu().numpy(),
                counts=counts.cpu().numpy(), err=int(err.item()))


def run_gpu_fused(case: dict, with_intermediates: bool = True) -> dict:
    """The one-kernel path (cluster of S CTAs per row)."""
    import dsa_sparse_indexer_gb300 as dsa
    cfg = case["cfg"]
    err = dsa.new_error_flags("cuda")
    r2q = None if case["r2q"] is None else dev(case["r2q"])
    S, R, K = cfg.S, cfg.rows, cfg.K
    g = Guards()
    o = dsa.indexer_fused(dev(case["local"]), dev(case["ends"]), K, cfg.I, dev(case["bt"]),
                          cfg.block_size, row_starts=dev(case["starts"]), row_to_req=r2q,
                          ids=g.empty((R, K), torch.int32), slots=g.empty((S, R, K), torch.int32),
                          counts=g.empty((S, R), torch.int32),
                          scores=g.empty((R, K), torch.float32),
                          local_idx=g.empty((S, R, K), torch.int32) if with_intermediates else None,
                          cand=g.empty((R, S * K, 2), torch.float32) if with_intermediates else None,
                          err_flags=err)
    g.check()
    got = dict(ids=o["ids"].cpu().numpy(), scores=o["scores"].cpu().numpy(),
               slots=o["slots"].cpu().numpy(), counts=o["counts"].cpu().numpy(),
               err=int(err.item()))
    if with_intermediates:
        c = o["cand"].cpu().numpy()
        got.update(local_idx=o["local_idx"].cpu().numpy(), cand_scores=c[..., 0],
                   cand_ids=c[..., 1].view(np.int32))
    return got


def run_oracle(case: dict, rows) -> dict:
    cfg = case["cfg"]
    return OP.run_rows(case["local"], case["starts"], case["ends"], cfg.S, cfg.I, cfg.K,
                       rows=rows, tables=case["bt"], row_to_req=case["r2q"],
                       block_size=cfg.block_size)


def bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def assert_indexer_parity(case: dict, got: dict, rows) -> None:
    """Bit-exact comparison of every indexer output on the listed rows."""
    cfg = case["cfg"]
    want = run_oracle(case, rows)
    rows = np.asarray(rows)
    assert got["err"] == 0
    if "local_idx" in got:
        np.testing.assert_array_equal(got["local_idx"][:, rows], want["local_idx"])
        np.testing.assert_array_equal(bits(got["cand_scores"][rows]), bits(want["cand_scores"]))
        np.testing.assert_array_equal(got["cand_ids"][rows], want["cand_ids"])
    np.testing.assert_array_equal(got["ids"][rows], want["ids"])
    # scores: value equality (-0.0 may come back as +0.0)
    np.testing.assert_array_equal(got["scores"][rows], want["scores"])
    np.testing.assert_array_equal(got["slots"][:, rows], want["slots"])
    np.testing.assert_array_equal(got["counts"][:, rows], want["counts"])
    # and the merged ids are the definition: top-K of the unsharded row
    for j, r in enumerate(rows):
        ref_ids, _ = OX.global_topk(case["x"][r], int(case["starts"][r]), int(case["ends"][r]),
                                    cfg.K)
        np.testing.assert_array_equal(got["ids"][r], ref_ids)
    return want


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(ref), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def combine_tolerance(ref: np.ndarray) -> np.ndarray:
    """bf16 output vs the oracle's unrounded fp64: 1e-2 absolute, widened to half
    a bf16 ulp (+ fp32 accumulation slack) where a bf16 ulp exceeds it."""
    return np.maximum(1e-2, 0.5 * bf16_ulp(ref) + 1e-5 * np.maximum(1.0, np.abs(ref)))


def assert_combine_parity(out_bf16: torch.Tensor, lse: torch.Tensor, part_bits: np.ndarray,
                          lse2: np.ndarray, rows) -> None:
    rows = np.asarray(rows)
    ref_out, ref_lse = OC.lse_combine(OC.bf16_to_f64(part_bits[:, rows]), lse2[:, rows])
    got = out_bf16.float().cpu().numpy()[rows].astype(np.float64)
    tol = combine_tolerance(ref_out)
    bad = np.abs(got - ref_out) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref_out[bad][:5])
    got_lse = lse.cpu().numpy()[rows].astype(np.float64)
    inf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), inf)
    d = np.abs(got_lse[~inf] - ref_lse[~inf])
    assert np.all(d <= 1e-5 * np.maximum(1.0, np.abs(ref_lse[~inf]))), d.max()


# ---------------------------------------------------------------------------
# Every row of a full-size workload against the oracle, over spawned host
# processes (spawned, not forked: the parent already holds a GPU context).
# Each worker rebuilds the workload from its seeds and compares its share of
# the rows; the definition check (a brute-force sort of the unsharded row) is
# left to the sampled rows of assert_indexer_parity.
# ---------------------------------------------------------------------------
_KEYS_S = ("local_idx", "slots", "counts")          # [S, rows, ...]
_KEYS_R = ("cand_scores", "cand_ids", "ids", "scores")   # [rows, ...]
_WORKER: dict = {}


def _rows_worker_init(name: str) -> None:
    case = make_case(name)
    case.pop("x")                      # only the shards' rows are read
    _WORKER["case"] = case


def _rows_worker_check(task):
    rows, got = task
    want = run_oracle(_WORKER["case"], rows)
    bad = {}
    for k in _KEYS_S + _KEYS_R:
        g, w = got[k], want[k]
        if k in ("cand_scores",):
            g, w = bits(g), bits(w)
        if not np.array_equal(g, w):
            diff = (g != w).reshape((len(rows), -1) if k in _KEYS_R else (g.shape[0], len(rows), -1))
            first = np.argwhere(diff.any(axis=-1))[0]
            bad[k] = int(rows[first[-1]])
    return len(rows), bad


def assert_all_rows_match_oracle(name: str, got: dict, procs: int | None = None) -> int:
    """Every row of workload `name` (as make_case builds it) bit-exact against
    the oracle's steps; returns the number of rows checked."""
    import multiprocessing as mp
    import os
    cfg = W.CONFIGS[name]
    n = procs or max(1, min(8, (os.cpu_count() or 2) - 1))
    chunks = np.array_split(np.arange(cfg.rows), 4 * n)
    tasks = []
    for c in chunks:
        sub = {k: np.ascontiguousarray(got[k][:, c]) for k in _KEYS_S}
        sub.update({k: np.ascontiguousarray(got[k][c]) for k in _KEYS_R})
        tasks.append((c, sub))
    checked = 0
    with mp.get_context("spawn").Pool(n, initializer=_rows_worker_init, initargs=(name,)) as pool:
        for cnt, bad in pool.imap_unordered(_rows_worker_check, tasks):
            assert not bad, f"first mismatching row per output: {bad}"
            checked += cnt
    assert checked == cfg.rows
    return checked
