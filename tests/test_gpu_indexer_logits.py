"""GPU parity of dsa_indexer_logits (fp8 tensor-core indexer logits) with the
fp64 oracle (oracle/indexer_logits.py), and of the indexer step it feeds.

Tolerance, from the arithmetic: products of two e4m3 values are exact in fp32;
each head's 128 products are summed by the tensor cores in fp32 (the
accumulation order and the width of the adder's alignment are the hardware's:
2^-13 of the sum of magnitudes covers an adder that keeps 14 bits), then the
ReLU'd head sums are weighted and summed in fp32 (64 rounded steps).  So
|gpu - oracle| <= 2^-13 * M + 1e-6 where M = sum_h |w_h| sum_d |q_hd k_d|
(oracle.indexer_logits.magnitude).  The top-K that follows decides indices
from the GPU's fp32 logits; its parity is checked on those same logits
(bit-exact), the oracle's steps applied to them.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import dcp_layout as OL
from oracle import indexer_logits as IL
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu

TOL_REL = 2.0 ** -13


def _case(S, I, rows, Lmax, bs, seed, reqs=None, ends=None, starts=None):
    rng = np.random.default_rng(seed)
    reqs = rows if reqs is None else reqs
    if ends is None:
        ends = rng.integers(1, Lmax + 1, rows).astype(np.int32)
    starts = np.zeros(rows, np.int32) if starts is None else starts
    ld = (max(OL.local_count(Lmax, s, S, I) for s in range(S)) + 3) // 4 * 4
    max_blocks = -(-ld // bs)
    n_slots = reqs * max_blocks * bs
    tables = np.stack([rng.permutation(reqs * max_blocks).astype(np.int32).reshape(reqs, -1)
                       for _ in range(S)])
    return dict(S=S, I=I, rows=rows, ld=ld, bs=bs, starts=starts, ends=ends, tables=tables,
                r2q=None if reqs == rows else np.zeros(rows, np.int32),
                q=W.indexer_query(rows, seed + 1), w=W.indexer_weights(rows, seed + 2),
                k=W.indexer_keys(S, n_slots, seed + 3))


def _run(c, fill=np.nan):
    import dsa_sparse_indexer_gb300 as dsa
    g = G.Guards()
    out = g.empty((c["S"], c["rows"], c["ld"]), torch.float32)
    out.fill_(fill)
    err = dsa.new_error_flags("cuda")
    dsa.indexer_logits(G.dev(c["q"]), G.dev(c["w"]), G.dev(c["k"]), G.dev(c["tables"]), c["bs"],
                       G.dev(c["ends"]), c["I"], c["ld"], row_starts=G.dev(c["starts"]),
                       row_to_req=None if c["r2q"] is None else G.dev(c["r2q"]), out=out,
                       err_flags=err)
    g.check()
    return out.cpu().numpy(), int(err.item())


def _check(c, got, rows=None):
    rows = np.arange(c["rows"]) if rows is None else np.asarray(rows)
    args = (c["q"], c["w"], c["k"], c["starts"], c["ends"], c["S"], c["I"], c["tables"], c["bs"])
    want = IL.shard_logits(*args, row_to_req=c["r2q"], ld=c["ld"], rows=rows)
    mag = IL.magnitude(*args, row_to_req=c["r2q"], ld=c["ld"], rows=rows)
    g = got[:, rows].astype(np.float64)
    inside = ~np.isnan(want)
    assert np.isnan(g[~inside]).all()                       # outside the range: untouched
    d = np.abs(g[inside] - want[inside])
    tol = TOL_REL * mag[inside] + 1e-6
    assert (d <= tol).all(), (d.max(), (d / np.maximum(mag[inside], 1e-30)).max())
    return float((d / np.maximum(mag[inside], 1e-30)).max())


@pytest.mark.parametrize("S,I,bs", [(1, 1, 64), (4, 1, 64), (3, 2, 16), (8, 4, 32), (2, 1, 128)])
def test_logits_match_the_oracle(S, I, bs):
    c = _case(S, I, rows=6, Lmax=S * 2600 + 37, bs=bs, seed=S * 100 + I)
    c["ends"][:3] = [S * 2600 + 37, 1, S * I * 3 + 1]         # longest, one token, a few
    c["starts"][4] = 129
    got, err = _run(c)
    assert err == 0
    _check(c, got)


def test_one_request_shared_by_all_rows():
    """Prefill-like: every row reads the same request's cache (row_to_req = 0)."""
    rows, S = 40, 4
    c = _case(S, 1, rows=rows, Lmax=4096, bs=64, seed=7, reqs=1,
              ends=(3000 + 24 * np.arange(rows)).astype(np.int32))
    got, err = _run(c)
    assert err == 0
    _check(c, got)


def test_bad_table_entries_read_zero_keys_and_set_the_bounds_flag():
    c = _case(2, 1, rows=2, Lmax=1000, bs=64, seed=9, ends=np.array([1000, 500], np.int32))
    c["tables"][0, 0, 1] = -5                      # shard 0, row 0, local block 1
    got, err = _run(c)
    assert err & 1
    good, _ = _run(dict(c, tables=np.abs(c["tables"])))
    # block 1 of shard 0, row 0 scored against zero keys: logits 0
    np.testing.assert_array_equal(got[0, 0, 64:128], 0.0)
    np.testing.assert_array_equal(got[0, 0, :64], good[0, 0, :64])
    np.testing.assert_array_equal(got[1], good[1])


def test_decode_workload_full_size_then_the_indexer_steps():
    """The decode batch at full size (64 rows, S = 4, up to 65536 tokens), on
    sampled rows; then the local top-K, merge and convert on the GPU's logits
    against the oracle's steps on the same logits (bit-exact)."""
    import dsa_sparse_indexer_gb300 as dsa
    cfg = W.CONFIGS["decode"]
    starts, ends = W.row_ranges(cfg)
    tables = W.block_tables(cfg)
    n_slots = cfg.reqs * cfg.max_blocks * cfg.block_size
    c = dict(S=cfg.S, I=cfg.I, rows=cfg.rows, ld=cfg.ld, bs=cfg.block_size, starts=starts,
             ends=ends, tables=tables, r2q=None, q=W.indexer_query(cfg.rows, 11),
             w=W.indexer_weights(cfg.rows, 12), k=W.indexer_keys(cfg.S, n_slots, 13))
    got, err = _run(c)
    assert err == 0
    rel = _check(c, got, rows=[0, 17, 40, 63])
    assert rel <= TOL_REL
    # the indexer steps on these logits
    local = np.nan_to_num(got, nan=0.0).astype(np.float32)
    case = dict(cfg=cfg, x=None, local=local, starts=starts, ends=ends, bt=tables, r2q=None)
    res = G.run_gpu(case)
    want = G.run_oracle(case, np.arange(cfg.rows))
    for k in ("local_idx", "ids", "slots", "counts"):
        np.testing.assert_array_equal(res[k], want[k])
    assert res["err"] == 0


def test_prefill_workload_full_size_grouped_rows():
    """The prefill batch at full size (4096 rows sharing one request, so the
    kernel takes eight rows an item, four per MMA pass): sampled rows of every
    shard against the oracle, including the first and last rows, rows at item
    boundaries and the rows whose ranges end inside a chunk."""
    cfg = W.CONFIGS["prefill"]
    starts, ends = W.row_ranges(cfg)
    tables = W.block_tables(cfg)
    n_slots = cfg.reqs * cfg.max_blocks * cfg.block_size
    c = dict(S=cfg.S, I=cfg.I, rows=cfg.rows, ld=cfg.ld, bs=cfg.block_size, starts=starts,
             ends=ends, tables=tables, r2q=np.zeros(cfg.rows, np.int32),
             q=W.indexer_query(cfg.rows, 41), w=W.indexer_weights(cfg.rows, 42),
             k=W.indexer_keys(cfg.S, n_slots, 43))
    got, err = _run(c)
    assert err == 0
    rows = [0, 1, 7, 8, 9, 1023, 2047, 2048, 3000, 4091, 4095]
    assert _check(c, got, rows=rows) <= TOL_REL


@pytest.mark.parametrize("S,I,bs,rows", [(3, 2, 64, 13), (8, 4, 32, 9), (2, 1, 16, 21),
                                         (4, 16, 128, 4)])
def test_grouped_rows_with_interleave_starts_and_a_partial_group(S, I, bs, rows):
    """Rows sharing one request (the grouped kernel: eight rows an item in two
    MMA passes of four) with interleave > 1, nonzero starts, a batch that is
    not a multiple of eight (the last item's missing rows read zero queries
    and write nothing), rows shorter than a tile and a row of one token."""
    rng = np.random.default_rng(S * 7 + rows)
    Lmax = S * I * 700 + 5
    ends = rng.integers(Lmax // 2, Lmax + 1, rows).astype(np.int32)
    ends[0], ends[-1] = Lmax, 1
    starts = np.zeros(rows, np.int32)
    starts[1::3] = rng.integers(0, 300, len(starts[1::3]))
    starts = np.minimum(starts, ends).astype(np.int32)
    c = _case(S, I, rows=rows, Lmax=Lmax, bs=bs, seed=S * 11 + rows, reqs=1, ends=ends,
              starts=starts)
    got, err = _run(c)
    assert err == 0
    assert _check(c, got) <= TOL_REL
