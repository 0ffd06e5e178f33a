"""Pins for the oracle's top-K, pack, merge and convert steps.

The central property (a consequence of the ranking being a total order): every
element of the global top-K is in its own shard's top-K, so merging the shards'
top-Ks reproduces the top-K of the whole, unsharded row.  It is checked against
a brute-force pure-Python sort on many small random rows with forced ties.
"""
import numpy as np
import pytest

from oracle import dcp_layout as L
from oracle import indexer as X
from oracle import pipeline as P


def brute_topk(x, st, en, K):
    """Pure-Python sort of (score, id) pairs: no numpy ordering involved."""
    items = sorted(range(st, en), key=lambda t: (-float(x[t]), t))[:K]
    return items + [-1] * (K - len(items))


def random_row(rng, n):
    kind = rng.integers(0, 4)
    if kind == 0:       # coarse grid: many ties, includes -0.0
        v = np.rint(rng.standard_normal(n) * 2) / 4
        v = np.where(rng.random(n) < 0.1, -0.0, v)
    elif kind == 1:     # very few distinct values
        v = rng.integers(-2, 3, n).astype(np.float64)
    elif kind == 2:     # continuous
        v = rng.standard_normal(n)
    else:               # with infinities
        v = rng.standard_normal(n)
        v[rng.random(n) < 0.15] = -np.inf
        v[rng.random(n) < 0.03] = np.inf
    return v.astype(np.float32)


def sharded_topk(x, st, en, S, I, K):
    Lmax = len(x)
    local = L.shard_rows(x[None, :], [en], S, I, ld=Lmax + 4)
    res = P.run_rows(local, np.array([st]), np.array([en]), S, I, K)
    return res


def test_global_topk_matches_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        n = int(rng.integers(0, 120))
        x = random_row(rng, n + 5)
        st = int(rng.integers(0, 5))
        en = st + n
        K = int(rng.integers(1, 40))
        ids, sc = X.global_topk(x, st, en, K)
        assert list(ids) == brute_topk(x, st, en, K)
        valid = ids >= 0
        assert np.array_equal(sc[valid].view(np.uint32), x[ids[valid]].view(np.uint32))
        assert np.all(np.isneginf(sc[~valid]))


def test_sharded_merge_equals_unsharded_topk():
    """>= 10^4 random small rows, S in 1..8, I in 1..5, K in 1..64."""
    rng = np.random.default_rng(2)
    checked = 0
    while checked < 10000:
        S = int(rng.integers(1, 9))
        I = int(rng.integers(1, 6))
        K = int(rng.integers(1, 65))
        Lmax = int(rng.integers(1, 301))
        x = random_row(rng, Lmax)
        en = int(rng.integers(0, Lmax + 1))
        st = int(rng.integers(0, en + 1)) if rng.random() < 0.3 else 0
        res = sharded_topk(x, st, en, S, I, K)
        want = brute_topk(x, st, en, K)
        assert list(res["ids"][0]) == want, (S, I, K, st, en)
        checked += 1


def test_single_shard_is_plain_sort():
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(1, 400))
        x = random_row(rng, n)
        K = int(rng.integers(1, 80))
        res = sharded_topk(x, 0, n, 1, 1, K)
        assert list(res["ids"][0]) == brute_topk(x, 0, n, K)
        # with one shard the local top-K is the sorted set of the same ids
        local = res["local_idx"][0, 0]
        assert sorted(t for t in brute_topk(x, 0, n, K) if t >= 0) == \
            [int(v) for v in local if v >= 0]


def test_ties_go_to_smaller_id_across_shards():
    # S=2, I=1: even ids on shard 0, odd on shard 1.  All scores equal.
    x = np.zeros(10, np.float32)
    res = sharded_topk(x, 0, 10, 2, 1, 4)
    assert list(res["ids"][0]) == [0, 1, 2, 3]
    x = np.array([1, 5, 5, 5, 1, 5, 0, 0], np.float32)
    res = sharded_topk(x, 0, 8, 2, 1, 3)
    assert list(res["ids"][0]) == [1, 2, 3]


def test_negative_zero_ties_with_positive_zero():
    x = np.array([-0.0, 0.0, -0.0, 0.0, -1.0], np.float32)
    for S in (1, 2, 3):
        res = sharded_topk(x, 0, 5, S, 1, 3)
        assert list(res["ids"][0]) == [0, 1, 2]
    x = np.array([0.0, -0.0, -0.0], np.float32)
    assert list(sharded_topk(x, 0, 3, 2, 1, 2)["ids"][0]) == [0, 1]


def test_neg_inf_is_selectable_and_padding_is_last():
    x = np.array([-np.inf, -np.inf, 3.0], np.float32)
    res = sharded_topk(x, 0, 3, 2, 1, 5)
    assert list(res["ids"][0]) == [2, 0, 1, -1, -1]
    assert np.isneginf(res["scores"][0][1:]).all()


def test_short_rows_pad_and_empty_shards():
    rng = np.random.default_rng(4)
    S, I, K = 8, 4, 16
    for en in range(0, 40):
        x = rng.standard_normal(64).astype(np.float32)
        res = sharded_topk(x, 0, en, S, I, K)
        ids = res["ids"][0]
        n_valid = min(K, en)
        assert np.all(ids[:n_valid] >= 0) and np.all(ids[n_valid:] == -1)
        for s in range(S):
            held = L.local_count(en, s, S, I)
            li = res["local_idx"][s, 0]
            assert np.count_nonzero(li >= 0) == min(held, K)
            if held == 0:
                assert np.all(li == -1)


def test_local_topk_is_ascending_and_pack_maps_back():
    rng = np.random.default_rng(6)
    S, I, K = 4, 3, 20
    x = random_row(rng, 500)
    res = sharded_topk(x, 0, 500, S, I, K)
    for s in range(S):
        li = res["local_idx"][s, 0]
        v = li[li >= 0]
        assert np.all(np.diff(v) > 0)
        gid = res["cand_ids"][0, s * K:(s + 1) * K]
        sc = res["cand_scores"][0, s * K:(s + 1) * K]
        ok = gid >= 0
        assert np.array_equal(ok, li >= 0)
        sh, sl = L.global_to_local(gid[ok], S, I)
        assert np.all(sh == s) and np.array_equal(sl, li[ok])
        assert np.array_equal(sc[ok].view(np.uint32), x[gid[ok]].view(np.uint32))
        assert np.all(np.isneginf(sc[~ok]))


def test_merge_output_is_ranked_and_dominates():
    rng = np.random.default_rng(7)
    for _ in range(300):
        C = int(rng.integers(1, 200))
        K = int(rng.integers(1, 60))
        sc = random_row(rng, C)
        ids = rng.permutation(1000)[:C].astype(np.int64)
        ids[rng.random(C) < 0.2] = -1
        sc[ids < 0] = -np.inf
        out, osc = X.merge(sc, ids, K)
        nvalid = int((ids >= 0).sum())
        m = min(K, nvalid)
        assert np.all(out[:m] >= 0) and np.all(out[m:] == -1)
        key = [(-float(v) + 0.0, int(t)) for v, t in zip(osc[:m], out[:m])]
        assert key == sorted(key)
        if m:
            worst = key[-1]
            chosen = set(out[:m].tolist())
            for v, t in zip(sc, ids):
                if t >= 0 and t not in chosen:
                    assert (-float(v) + 0.0, int(t)) > worst


def test_convert_identity_table_and_inverse():
    rng = np.random.default_rng(8)
    S, I, K, bs = 4, 2, 64, 8
    reqs, max_blocks = 3, 40
    ident = np.arange(reqs * max_blocks).reshape(reqs, max_blocks)
    tables = np.broadcast_to(ident, (S, reqs, max_blocks))
    perm = np.stack([rng.permutation(reqs * max_blocks).reshape(reqs, max_blocks)
                     for _ in range(S)])
    for trial in range(50):
        q = int(rng.integers(0, reqs))
        n = int(rng.integers(0, K + 1))
        ids = np.full(K, -1, np.int64)
        ids[:n] = rng.permutation(S * I * max_blocks * bs // 2)[:n]
        slots, counts, err = X.convert_compact(ids, S, I, tables[:, q], bs)
        assert not err
        assert counts.sum() == n
        sh, loc = L.global_to_local(ids[:n], S, I) if n else (np.array([]), np.array([]))
        for s in range(S):
            c = int(counts[s])
            assert np.all(slots[s, c:] == -1)
            mine = loc[sh == s]
            # identity table: slot = req * max_blocks * bs + local slot
            assert np.array_equal(slots[s, :c], q * max_blocks * bs + mine)
        # random table: invert the table and recover the ids, in merged order
        slots, counts, err = X.convert_compact(ids, S, I, perm[:, q], bs)
        assert not err
        for s in range(S):
            c = int(counts[s])
            inv = {int(b): col for col, b in enumerate(perm[s, q])}
            back_local = [inv[int(v) // bs] * bs + int(v) % bs for v in slots[s, :c]]
            back = L.local_to_global(s, np.array(back_local, np.int64), S, I) if c else []
            assert list(back) == [int(t) for t in ids[:n] if L.owner(t, S, I) == s]


def test_convert_flags_out_of_range_blocks():
    S, I, bs = 2, 1, 4
    tables = np.array([[0, 1], [2, -1]])          # shard 1, column 1 unallocated
    ids = np.array([0, 1, 2, 3, 9, 17, -1, -1])   # id 17 -> shard 1, slot 8, col 2
    slots, counts, err = X.convert_compact(ids, S, I, tables, bs)
    assert err
    assert list(counts) == [2, 4]
    assert list(slots[0, :2]) == [0, 1]
    # id 1 -> slot 0, id 3 -> slot 1 (block 2); id 9 -> local 4 -> col 1 (-1); 17 -> col 4
    assert list(slots[1, :4]) == [8, 9, -1, -1]
