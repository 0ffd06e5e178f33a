"""Pins of the write-side slot-mapping oracle (oracle/kv_write.py) against a
hand-worked example, the plain paged-cache mapping it reduces to without
sharding, the read side (the merged-id conversion must find each token where
the write side put it), the inverse walk through the block tables, and its
error cases."""
import numpy as np
import pytest

from oracle import dcp_layout as OL
from oracle import indexer as OX
from oracle import kv_write as KW


def test_worked_example_two_shards_interleave_two():
    """S = 2, I = 2, block size 4, one request.  Shard 0 holds tokens 0, 1, 4,
    5, 8, 9 (local slots 0..5) in blocks 5 then 9; shard 1 holds 2, 3, 6, 7,
    10, 11 in blocks 2 then 7 (worked by hand from the ownership rule)."""
    tables = np.array([[[5, 9]], [[2, 7]]])
    got, err = KW.slot_mapping(np.arange(12), np.zeros(12), 2, 2, tables, 4)
    assert not err
    np.testing.assert_array_equal(
        got[0], [20, 21, -1, -1, 22, 23, -1, -1, 36, 37, -1, -1])
    np.testing.assert_array_equal(
        got[1], [-1, -1, 8, 9, -1, -1, 10, 11, -1, -1, 28, 29])


def test_one_shard_is_the_plain_paged_mapping():
    """Without sharding a token at position t of request q goes to
    table[q][t // bs] * bs + t % bs."""
    rng = np.random.default_rng(1)
    bs, reqs, width = 16, 5, 12
    tables = rng.permutation(reqs * width).reshape(1, reqs, width)
    pos = rng.integers(0, bs * width, 300)
    req = rng.integers(0, reqs, 300)
    got, err = KW.slot_mapping(pos, req, 1, 1, tables, bs)
    assert not err
    np.testing.assert_array_equal(got[0], tables[0, req, pos // bs] * bs + pos % bs)


def _random_case(rng, S, I, bs, reqs=6, L=700):
    width = -(-OL.local_count(L, 0, S, I) // bs) + 1
    tables = np.stack([rng.permutation(reqs * width).reshape(reqs, width) for _ in range(S)])
    lens = rng.integers(1, L + 1, reqs)
    return tables, lens


@pytest.mark.parametrize("S,I,bs", [(2, 1, 4), (4, 3, 16), (3, 5, 8), (8, 2, 64)])
def test_read_side_finds_what_the_write_side_wrote(S, I, bs):
    """Write every token of each request, then convert a merged id list of that
    request: each shard's compacted slots are exactly the written slots of its
    tokens, in merged order."""
    rng = np.random.default_rng(S * 100 + I * 10 + bs)
    tables, lens = _random_case(rng, S, I, bs)
    for q, L in enumerate(lens):
        written, err = KW.slot_mapping(np.arange(L), np.full(L, q), S, I, tables, bs)
        assert not err
        merged = rng.permutation(L)[:min(L, 64)]
        slots, counts, err2 = OX.convert_compact(merged, S, I, tables[:, q], bs)
        assert not err2
        for s in range(S):
            mine = [written[s, t] for t in merged if written[s, t] >= 0]
            assert counts[s] == len(mine)
            np.testing.assert_array_equal(slots[s, :counts[s]], mine)


@pytest.mark.parametrize("S,I,bs", [(2, 1, 4), (4, 3, 16), (5, 2, 8)])
def test_inverse_walk_and_one_owner(S, I, bs):
    """Every token is stored on exactly one shard; walking its slot back
    through that shard's table (which block column holds the slot's block) and
    the local-to-global map gives the token and its request; no two tokens
    share a slot on a shard."""
    rng = np.random.default_rng(7 + S + I + bs)
    tables, lens = _random_case(rng, S, I, bs)
    pos = np.concatenate([np.arange(L) for L in lens])
    req = np.concatenate([np.full(L, q) for q, L in enumerate(lens)])
    got, err = KW.slot_mapping(pos, req, S, I, tables, bs)
    assert not err
    assert ((got >= 0).sum(axis=0) == 1).all()
    for s in range(S):
        held = np.flatnonzero(got[s] >= 0)
        assert len(np.unique(got[s, held])) == len(held)
        for i in held:
            p = got[s, i]
            q, col = np.argwhere(tables[s] == p // bs)[0]
            l = col * bs + p % bs
            assert q == req[i]
            assert OL.local_to_global(s, np.array([l]), S, I)[0] == pos[i]


def test_padding_and_errors():
    tables = np.array([[[3, -1]], [[4, 6]]])
    # padding token, request out of range, column past the width, negative entry
    pos = np.array([-1, 0, 40, 4])
    req = np.array([0, 1, 0, 0])
    got, err = KW.slot_mapping(pos, req, 2, 2, tables, 2)
    assert err
    assert (got == -1).all()
    got, err = KW.slot_mapping(np.array([-5, 3]), np.array([0, 0]), 2, 2, tables, 2)
    assert not err
    np.testing.assert_array_equal(got, [[-1, -1], [-1, 9]])
    big = np.array([[[2 ** 30]]])
    got, err = KW.slot_mapping(np.array([1]), np.array([0]), 1, 1, big, 4)
    assert err and got[0, 0] == -1
