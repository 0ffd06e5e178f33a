"""GPU parity of the write-side slot mapping (dsa_slot_mapping) with the oracle
(oracle/kv_write.py), element by element, on the workloads' block tables: the
new token of every decode row, a whole prefill chunk, every token of sampled
requests, and the edge cases (padding tokens, bad requests, columns and table
entries, more shards than a cluster holds, block sizes that are not powers of
two).  Also: the read side (dsa_convert_index_compact) finds each merged id
where the write side put it."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kv_write as KW
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu


def _run(pos, req, S, I, bt, bs):
    import dsa_sparse_indexer_gb300 as dsa
    err = dsa.new_error_flags("cuda")
    g = G.Guards()
    out = dsa.slot_mapping(G.dev(np.asarray(pos, np.int32)), G.dev(bt), bs, I,
                           token_req=None if req is None else G.dev(np.asarray(req, np.int32)),
                           out=g.empty((S, len(pos)), torch.int32), err_flags=err)
    g.check()
    return out.cpu().numpy(), int(err.item())


def _check(pos, req, S, I, bt, bs):
    got, err = _run(pos, req, S, I, bt, bs)
    want, werr = KW.slot_mapping(pos, np.arange(len(pos)) if req is None else req, S, I, bt, bs)
    np.testing.assert_array_equal(got, want)
    assert bool(err) == werr
    return got


@pytest.mark.parametrize("name", ["tiny", "decode", "long_decode", "prefill", "ragged"])
def test_new_tokens_of_every_workload(name):
    cfg = W.CONFIGS[name]
    _, ends = W.row_ranges(cfg)
    bt = W.block_tables(cfg)
    r2q = G.row_to_req_for(cfg)
    if r2q is None:       # decode-like: the last token of every row, row r = request r
        pos = np.maximum(ends.astype(np.int64) - 1, -1)
        _check(pos, None, cfg.S, cfg.I, bt, cfg.block_size)
    else:                 # prefill chunk: one request, the chunk's own tokens
        pos = np.arange(int(ends.min()) - 1, int(ends.max()))
        _check(pos, np.zeros(len(pos), np.int64), cfg.S, cfg.I, bt, cfg.block_size)


@pytest.mark.parametrize("name", ["decode", "long_decode", "ragged"])
def test_every_token_of_sampled_requests(name):
    cfg = W.CONFIGS[name]
    _, ends = W.row_ranges(cfg)
    bt = W.block_tables(cfg)
    rng = np.random.default_rng(3)
    qs = rng.choice(cfg.rows, 3, replace=False)
    pos = np.concatenate([np.arange(int(ends[q])) for q in qs])
    req = np.concatenate([np.full(int(ends[q]), q) for q in qs])
    got = _check(pos, req, cfg.S, cfg.I, bt, cfg.block_size)
    held = got >= 0
    assert (held.sum(axis=0) == 1).all()
    for s in range(cfg.S):
        assert len(np.unique(got[s, held[s]])) == held[s].sum()


@pytest.mark.parametrize("S,I,bs", [(16, 3, 48), (5, 7, 10), (1, 1, 64), (64, 1, 16)])
def test_shapes_padding_and_bad_entries(S, I, bs):
    rng = np.random.default_rng(S + I + bs)
    reqs, width = 7, 9
    bt = np.stack([rng.permutation(reqs * width).reshape(reqs, width) for _ in range(S)])
    bt = bt.astype(np.int32)
    n = 3000
    pos = rng.integers(0, S * I * bs * width, n)
    req = rng.integers(0, reqs, n)
    _check(pos, req, S, I, bt, bs)                       # every token valid
    pos[::97] = -1                                       # padding tokens: no error
    _check(pos, req, S, I, bt, bs)
    bad = bt.copy()
    bad[:, 2, 4] = -5                                    # negative table entries
    req2 = req.copy()
    req2[5] = reqs                                       # request out of range
    pos2 = pos.copy()
    pos2[7] = S * I * bs * width + 3                     # column past the width
    _check(pos2, req2, S, I, bad, bs)


def test_read_side_finds_what_the_write_side_wrote():
    """Merged ids of the tiny and ragged workloads, mapped by the convert
    kernel, are the slots the write side gives those tokens, shard by shard in
    merged order."""
    for name in ("tiny", "ragged"):
        case = G.make_case(name)
        cfg = case["cfg"]
        got = G.run_gpu(case)
        assert got["err"] == 0
        ids = got["ids"]
        r2q = case["r2q"]
        for r in range(min(cfg.rows, 32)):
            q = r if r2q is None else int(r2q[r])
            valid = ids[r][ids[r] >= 0]
            written, err = _run(valid, np.full(len(valid), q), cfg.S, cfg.I, case["bt"],
                                cfg.block_size)
            assert err == 0
            for s in range(cfg.S):
                mine = written[s][written[s] >= 0]
                n = got["counts"][s, r]
                assert n == len(mine)
                np.testing.assert_array_equal(got["slots"][s, r, :n], mine)
