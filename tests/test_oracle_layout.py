"""Pins for the oracle's DCP layout (ownership, local slots, local lengths).

The oracle derives everything by counting from the ownership rule; these tests
check it against the worked example printed on the PR #46076 page, against
independently derived closed forms, and against invariants.
"""
import json
import os

import numpy as np
import pytest

from oracle import dcp_layout as L

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (2, 2), (4, 4), (8, 4), (8, 16),
         (3, 5), (5, 3), (16, 2)]


def test_worked_example_localize_after_expand():
    """PR #46076 review highlights: expand per token, then localize -> [4,4,5]."""
    with open(os.path.join(HERE, "golden", "dcp_localize_worked_example.json")) as f:
        ex = json.load(f)
    S, s, I = ex["world_size"], ex["rank"], ex["interleave"]
    Lreq, q = ex["request_len"], ex["query_len"]
    per_token_global = [Lreq - q + 1 + j for j in range(q)]
    right = [L.local_count(g, s, S, I) for g in per_token_global]
    assert right == ex["expected_local_lens"]
    # The order the page calls wrong: localize the request length, then expand.
    loc_req = L.local_count(Lreq, s, S, I)
    wrong = [loc_req - (q - 1 - j) for j in range(q)]
    assert wrong == ex["wrong_order_local_lens"]
    assert right != wrong


@pytest.mark.parametrize("S,I", CASES)
def test_round_trip_global_local_global(S, I):
    t = np.arange(1 << 15, dtype=np.int64)
    s, slot = L.global_to_local(t, S, I)
    back = np.empty_like(t)
    for shard in range(S):
        sel = s == shard
        back[sel] = L.local_to_global(shard, slot[sel], S, I)
    assert np.array_equal(back, t)


@pytest.mark.parametrize("S,I", CASES)
def test_local_slots_are_a_bijection_and_counts_sum(S, I):
    rng = np.random.default_rng(S * 100 + I)
    for Ln in list(rng.integers(0, 3000, 20)) + [0, 1, I * S - 1, I * S, I * S + 1]:
        Ln = int(Ln)
        total = 0
        for shard in range(S):
            toks = L.owned_tokens(Ln, shard, S, I)
            n = L.local_count(Ln, shard, S, I)
            assert len(toks) == n
            if n:
                s_, slot = L.global_to_local(toks, S, I)
                assert np.all(s_ == shard)
                assert np.array_equal(slot, np.arange(n))
            total += n
        assert total == Ln


def _closed_form_count(Ln, s, S, I):
    # Derived by hand: every full round of I*S tokens gives each shard I tokens;
    # the partial round gives shard s the part of [s*I, s*I + I) below Ln mod I*S.
    full, rem = divmod(Ln, I * S)
    return full * I + min(max(rem - s * I, 0), I)


def _closed_form_slot(t, S, I):
    return (t // (I * S)) * I + t % I


def _closed_form_global(s, l, S, I):
    return (l // I) * (I * S) + s * I + l % I


@pytest.mark.parametrize("S,I", CASES)
def test_counting_matches_closed_forms(S, I):
    Ls = np.arange(0, 4 * I * S + 7)
    for shard in range(S):
        got = L.local_counts(Ls, shard, S, I)
        want = [_closed_form_count(int(x), shard, S, I) for x in Ls]
        assert list(got) == want
    t = np.arange(5000, dtype=np.int64)
    s, slot = L.global_to_local(t, S, I)
    assert np.array_equal(slot, _closed_form_slot(t, S, I))
    for shard in range(S):
        l = np.arange(300)
        assert np.array_equal(L.local_to_global(shard, l, S, I),
                              _closed_form_global(shard, l, S, I))


def test_shard_rows_places_each_token_at_its_local_slot():
    rng = np.random.default_rng(5)
    S, I, Lmax = 3, 4, 200
    x = rng.standard_normal((5, Lmax)).astype(np.float32)
    ends = np.array([200, 17, 0, 12, 199])
    ld = 72
    out = L.shard_rows(x, ends, S, I, ld, fill=np.nan)
    for r in range(5):
        for t in range(Lmax):
            s, l = L.global_to_local(np.array([t]), S, I)
            v = out[int(s[0]), r, int(l[0])]
            if t < ends[r]:
                assert v == x[r, t]
            else:
                assert np.isnan(v)
