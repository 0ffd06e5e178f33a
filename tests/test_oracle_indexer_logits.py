"""Pins of the indexer-logits oracle (oracle/indexer_logits.py), each against
something other than the oracle itself: the fp8 e4m3 format's published
values and PyTorch's own e4m3 conversion, closed forms of the ReLU-weighted
head sum, a pure-Python brute force, the linearity in the head weights that
the definition implies (ReLU before the weights), and the DCP identity: the
shards' logits over their paged local slots are the unsharded logits of the
tokens they own.

Plausible mistakes each of these catches: a wrong exponent bias or a missing
subnormal (decode values), ReLU applied after the weighted sum (linearity),
a transposed operand or a dropped head (brute force), a wrong block-table
lookup or ownership rule (the DCP identity)."""
import numpy as np
import pytest

import workloads as W
from oracle import dcp_layout as OL
from oracle import indexer_logits as IL


def test_e4m3_published_values():
    # OCP 8-bit floating point E4M3: bias 7, max normal 448, min subnormal 2^-9.
    cases = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x3C: 1.5, 0x30: 0.5}
    got = IL.e4m3_to_f64(np.array(list(cases), np.uint8))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))
    assert np.isnan(IL.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()
    assert np.array_equal(IL.e4m3_to_f64(np.array([0x80], np.uint8)), [0.0])   # -0


def test_e4m3_matches_torch_for_every_code():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = IL.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])


def test_one_hot_query_reads_one_key_entry_through_relu():
    rng = np.random.default_rng(0)
    H, d, n = 4, 128, 50
    keys = rng.standard_normal((n, d))
    for i in (0, 17, 127):
        q = np.zeros((H, d))
        q[2, i] = 1.0
        w = np.array([0.0, 0.0, 1.0, 0.0])
        np.testing.assert_array_equal(IL.logits(q, w, keys), np.maximum(keys[:, i], 0.0))
        # a negative head weight flips the sign of that head's (ReLU'd) share
        np.testing.assert_array_equal(IL.logits(q, -3.0 * w, keys),
                                      -3.0 * np.maximum(keys[:, i], 0.0))


def test_brute_force_small():
    rng = np.random.default_rng(1)
    H, d, n = 3, 5, 7
    q = rng.standard_normal((H, d))
    w = rng.standard_normal(H)
    keys = rng.standard_normal((n, d))
    want = []
    for u in range(n):
        tot = 0.0
        for h in range(H):
            dot = 0.0
            for c in range(d):
                dot += q[h][c] * keys[u][c]
            tot += w[h] * (dot if dot > 0 else 0.0)
        want.append(tot)
    np.testing.assert_allclose(IL.logits(q, w, keys), want, rtol=1e-13, atol=1e-13)


def test_linear_in_the_head_weights_not_in_the_queries():
    rng = np.random.default_rng(2)
    H, d, n = 8, 16, 40
    q = rng.standard_normal((H, d))
    keys = rng.standard_normal((n, d))
    w1, w2 = rng.standard_normal(H), rng.standard_normal(H)
    np.testing.assert_allclose(IL.logits(q, w1 + w2, keys),
                               IL.logits(q, w1, keys) + IL.logits(q, w2, keys), atol=1e-12)
    # ReLU per head: flipping the queries does not flip the logits
    a, b = IL.logits(q, w1, keys), IL.logits(-q, w1, keys)
    assert not np.allclose(a, -b)
    np.testing.assert_allclose(a + b, w1 @ np.abs(q @ keys.T), atol=1e-12)


@pytest.mark.parametrize("S,I,bs", [(1, 1, 16), (4, 1, 64), (3, 2, 8), (8, 4, 16)])
def test_shards_score_exactly_the_tokens_they_own(S, I, bs):
    """Global keys laid into per-shard paged caches by the ownership rule and
    random block tables: each shard's logit at local slot l is the unsharded
    logit of global token glob(s, l)."""
    rng = np.random.default_rng(S * 10 + I)
    R, H, d = 3, 4, 8
    L = 3 * S * I * bs + 5
    ends = np.array([L, L - 7, S * I + 1], np.int32)
    starts = np.array([0, 3, 0], np.int32)
    max_blocks = -(-max(OL.local_count(L, s, S, I) for s in range(S)) // bs)
    tables = np.stack([rng.permutation(R * max_blocks).astype(np.int32).reshape(R, max_blocks)
                       for _ in range(S)])
    n_slots = R * max_blocks * bs
    q = W.e4m3_codes(rng, (R, H, d))
    w = rng.standard_normal((R, H)).astype(np.float32)
    gkeys = W.e4m3_codes(rng, (R, L, d))             # request r's key of token t
    cache = np.zeros((S, n_slots, d), np.uint8)
    for r in range(R):
        s_of, l_of = OL.global_to_local(np.arange(L), S, I)
        for t in range(L):
            s, l = int(s_of[t]), int(l_of[t])
            cache[s, tables[s, r, l // bs] * bs + l % bs] = gkeys[r, t]
    got = IL.shard_logits(q, w, cache, starts, ends, S, I, tables, bs)
    for r in range(R):
        full = IL.logits(IL.e4m3_to_f64(q[r]), w[r], IL.e4m3_to_f64(gkeys[r]))
        for s in range(S):
            lo = OL.local_count(int(starts[r]), s, S, I)
            hi = OL.local_count(int(ends[r]), s, S, I)
            glob = OL.local_to_global(s, np.arange(lo, hi), S, I)
            np.testing.assert_array_equal(got[s, r, lo:hi], full[glob])
            assert np.isnan(got[s, r, :lo]).all() and np.isnan(got[s, r, hi:]).all()


def test_magnitude_bounds_every_logit():
    rng = np.random.default_rng(5)
    S, I, bs, R = 2, 1, 16, 2
    tables = np.arange(S * R * 4, dtype=np.int32).reshape(S, R, 4)
    q = W.e4m3_codes(rng, (R, 64, 128))
    w = rng.standard_normal((R, 64)).astype(np.float32)
    keys = W.e4m3_codes(rng, (S, S * R * 4 * bs, 128))   # every block the tables name
    ends = np.array([100, 77], np.int32)
    starts = np.zeros(R, np.int32)
    lg = IL.shard_logits(q, w, keys, starts, ends, S, I, tables, bs, fill=0.0)
    mag = IL.magnitude(q, w, keys, starts, ends, S, I, tables, bs)
    assert (np.abs(lg) <= mag + 1e-9).all() and (mag > 0).any()
