"""Pins of the PCP prefill oracle (oracle/pcp_prefill.py) against closed forms
and library routines: the RMS norm's unit RMS and scale invariance, the
interleaved rotation as complex multiplication (numpy complex arithmetic),
angle composition and norm preservation, the identity at position 0, and the
gather-then-insert round trip.

Plausible mistakes each catches: a missing square root or mean (unit RMS), a
sign flipped in the rotation or the pairs taken as (i, i + n) halves instead
of adjacent values (complex multiplication), cos and sin swapped (position 0
identity), a slot of -1 written (round trip)."""
import numpy as np
import pytest

from oracle import pcp_prefill as PP


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 512))
    y = PP.rms_norm(x, np.ones(512), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(PP.rms_norm(7.5 * x, np.ones(512), 0.0), y, rtol=1e-13)
    w = rng.standard_normal(512)
    np.testing.assert_allclose(PP.rms_norm(x, w, 0.0), y * w, rtol=1e-13)
    a, eps = 0.25, 1e-3                      # a constant row: a / sqrt(a^2 + eps)
    np.testing.assert_allclose(PP.rms_norm(np.full((1, 8), a), np.ones(8), eps),
                               a / np.sqrt(a * a + eps), rtol=1e-14)


def test_interleaved_rotation_is_complex_multiplication():
    rng = np.random.default_rng(1)
    T, n = 7, 32
    x = rng.standard_normal((T, 2 * n))
    ang = rng.uniform(-np.pi, np.pi, (T, n))
    got = PP.rope_interleaved(x, np.cos(ang), np.sin(ang))
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * ang)
    np.testing.assert_allclose(got[:, 0::2], z.real, atol=1e-13)
    np.testing.assert_allclose(got[:, 1::2], z.imag, atol=1e-13)
    # norm of every pair preserved; two rotations compose
    np.testing.assert_allclose(np.hypot(got[:, 0::2], got[:, 1::2]),
                               np.hypot(x[:, 0::2], x[:, 1::2]), rtol=1e-13)
    ang2 = rng.uniform(-np.pi, np.pi, (T, n))
    twice = PP.rope_interleaved(got, np.cos(ang2), np.sin(ang2))
    once = PP.rope_interleaved(x, np.cos(ang + ang2), np.sin(ang + ang2))
    np.testing.assert_allclose(twice, once, atol=1e-12)


def test_fused_norm_rope_position_zero_is_the_identity_rotation():
    rng = np.random.default_rng(2)
    T, d_c, d_r, P = 4, 512, 64, 100
    kv, kpe = rng.standard_normal((T, d_c)), rng.standard_normal((T, d_r))
    inv_freq = 10000.0 ** (-np.arange(0, d_r, 2) / d_r)
    ang = np.arange(P)[:, None] * inv_freq[None, :]
    cache = np.concatenate([np.cos(ang), np.sin(ang)], axis=1)
    w = rng.standard_normal(d_c)
    kv_o, kpe_o = PP.fused_norm_rope(kv, kpe, w, 1e-6, np.zeros(T, int), cache)
    np.testing.assert_allclose(kpe_o, kpe, atol=1e-15)
    np.testing.assert_allclose(kv_o, PP.rms_norm(kv, w, 1e-6), rtol=1e-15)
    pos = np.array([1, 17, 63, 99])
    _, kpe_p = PP.fused_norm_rope(kv, kpe, w, 1e-6, pos, cache)
    z = (kpe[:, 0::2] + 1j * kpe[:, 1::2]) * np.exp(1j * ang[pos])
    np.testing.assert_allclose(kpe_p[:, 0::2], z.real, atol=1e-12)
    np.testing.assert_allclose(kpe_p[:, 1::2], z.imag, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 8])
def test_gather_then_insert_round_trip(P):
    rng = np.random.default_rng(3 + P)
    T, d, n_slots = 40 * P + 3, 9, 1000
    rows = rng.standard_normal((T, d))
    cuts = np.linspace(0, T, P + 1).astype(int)
    gathered = PP.gather_ranks([rows[cuts[p]:cuts[p + 1]] for p in range(P)])
    np.testing.assert_array_equal(gathered, rows)
    slots = rng.permutation(n_slots)[:T]
    slots[::7] = -1                               # padding tokens write nothing
    cache0 = rng.standard_normal((n_slots, d))
    cache = PP.cache_insert(cache0, gathered, slots)
    keep = slots >= 0
    np.testing.assert_array_equal(cache[slots[keep]], rows[keep])
    untouched = np.setdiff1d(np.arange(n_slots), slots[keep])
    np.testing.assert_array_equal(cache[untouched], cache0[untouched])
