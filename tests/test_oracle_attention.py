"""Pins of the sparse MLA decode oracle (oracle/attention.py): closed forms
(one token, identical keys, one dominant score, no token) and the identity
that makes DCP work: the shards' partial attentions merged by the LSE combine
oracle equal one softmax attention over all the selected tokens (computed
here with scipy's logsumexp and softmax over the whole set)."""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as OA
from oracle import combine as OC

LN2 = np.log(2.0)


def test_one_token_returns_its_value_and_score():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((5, 24))
    k = rng.standard_normal((1, 24))
    out, lse2 = OA.sparse_mla_decode(q, k, 0.3, 16)
    np.testing.assert_allclose(out, np.broadcast_to(k[0, :16], (5, 16)), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse2, 0.3 * (q @ k[0]) / LN2, rtol=1e-15, atol=1e-15)


def test_identical_keys_average_the_values():
    """Equal keys give equal weights: the plain mean of the values and
    lse = s + ln n."""
    rng = np.random.default_rng(1)
    n, d_qk, d_v = 7, 20, 12
    rows = rng.standard_normal((n, d_qk))
    rows[:, d_v:] = rows[0, d_v:]                   # same rope part ...
    q = rng.standard_normal((3, d_qk))
    q[:, :d_v] = 0.0                                # ... and only it is scored
    out, lse2 = OA.sparse_mla_decode(q, rows, 0.7, d_v)
    np.testing.assert_allclose(out, np.broadcast_to(rows[:, :d_v].mean(0), (3, d_v)),
                               rtol=1e-14, atol=1e-14)
    s = 0.7 * (q @ rows[0])
    np.testing.assert_allclose(lse2, (s + np.log(n)) / LN2, rtol=1e-14)


def test_a_dominant_score_selects_its_value_without_overflow():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((6, 8))
    q = np.zeros((1, 8))
    q[0, 7] = 1.0
    rows[:, 7] = [1.0, 2.0, 900.0, 3.0, -5.0, 0.0]   # scores up to 900 * scale
    out, lse2 = OA.sparse_mla_decode(q, rows, 1.0, 4)
    np.testing.assert_allclose(out[0], rows[2, :4], rtol=0, atol=1e-300)
    np.testing.assert_allclose(lse2[0], 900.0 / LN2, rtol=1e-15)
    assert np.isfinite(out).all()


def test_no_token():
    out, lse2 = OA.sparse_mla_decode(np.ones((2, 8)), np.zeros((0, 8)), 1.0, 4)
    assert (out == 0).all() and np.isneginf(lse2).all()


@pytest.mark.parametrize("S,n", [(1, 40), (4, 300), (8, 97)])
def test_shards_combined_by_lse_equal_attention_over_all_tokens(S, n):
    """Split n selected tokens over S shards (some possibly empty), attend per
    shard, merge with the combine oracle: the result is softmax attention over
    all n tokens, to fp64 rounding."""
    rng = np.random.default_rng(S * 1000 + n)
    H, d_qk, d_v, scale = 6, 40, 32, 1 / np.sqrt(12.0)
    rows = rng.standard_normal((n, d_qk))
    q = rng.standard_normal((H, d_qk))
    owner = rng.integers(0, S, n)
    if S > 2:
        owner[owner == 1] = 0                          # shard 1 left empty
    parts, lses = [], []
    for s in range(S):
        o, l2 = OA.sparse_mla_decode(q, rows[owner == s], scale, d_v)
        parts.append(o)
        lses.append(l2)
    out, lse = OC.lse_combine(np.stack(parts), np.stack(lses))
    scores = scale * (q @ rows.T)
    want = softmax(scores, axis=1) @ rows[:, :d_v]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, logsumexp(scores, axis=1), rtol=1e-12, atol=1e-12)


def test_shard_attention_walks_each_shards_compacted_slots():
    """The per-(shard, row) driver reads exactly slots[s, r, :counts[s, r]]:
    slots past the count (here pointing at a poisoned row) never enter."""
    rng = np.random.default_rng(5)
    S, R, H, d_qk, d_v, n_slots, K = 2, 3, 2, 16, 8, 50, 6
    cache = rng.standard_normal((S, n_slots, d_qk))
    cache[:, 0] = 1e300
    q = rng.standard_normal((R, H, d_qk))
    slots = rng.integers(1, n_slots, (S, R, K))
    counts = np.array([[6, 2, 0], [3, 5, 1]])
    for s in range(S):
        for r in range(R):
            slots[s, r, counts[s, r]:] = 0
    out, lse2 = OA.shard_attention(q, cache, slots, counts, 0.5, d_v)
    for s in range(S):
        for r in range(R):
            o, l2 = OA.sparse_mla_decode(q[r], cache[s, slots[s, r, :counts[s, r]]], 0.5, d_v)
            np.testing.assert_array_equal(out[s, r], o)
            np.testing.assert_array_equal(lse2[s, r], l2)
    assert np.isneginf(lse2[0, 2]).all() and (out[0, 2] == 0).all()
