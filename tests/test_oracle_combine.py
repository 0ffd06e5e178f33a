"""Pins for the oracle's LSE combine.

The strongest pin: split a small attention problem across shards by the DCP
ownership rule, give each shard its own softmax-attention output and base-2
LSE, and require the combine to equal full softmax attention over the whole
sequence (computed here directly, with scipy's logsumexp for the LSE).
"""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import combine as C
from oracle import dcp_layout as L


def shard_partials(z, V, S, I):
    n = len(z)
    owner = L.owner(np.arange(n), S, I)
    O = np.zeros((S, V.shape[1]))
    lse2 = np.full(S, -np.inf)
    for s in range(S):
        m = owner == s
        if m.any():
            p = softmax(z[m])
            O[s] = p @ V[m]
            lse2[s] = logsumexp(z[m]) / np.log(2.0)     # base-2, as the kernel reports
    return O, lse2


@pytest.mark.parametrize("S,I,n", [(2, 1, 4096), (4, 1, 1000), (8, 4, 3000),
                                   (8, 16, 100), (3, 5, 7), (8, 4, 9), (1, 1, 50)])
def test_combine_equals_full_softmax_attention(S, I, n):
    rng = np.random.default_rng(S * 1000 + I * 10 + n)
    z = rng.standard_normal(n) * 3
    V = rng.standard_normal((n, 16))
    O, lse2 = shard_partials(z, V, S, I)
    out, lse = C.lse_combine(O, lse2)
    ref = softmax(z) @ V
    assert np.max(np.abs(out - ref)) < 1e-12
    assert abs(lse - logsumexp(z)) < 1e-12


def test_single_nonempty_shard_passes_through():
    rng = np.random.default_rng(1)
    O = rng.standard_normal((4, 3, 8))
    lse2 = np.full((4, 3), -np.inf)
    lse2[2] = [1.5, -3.0, 19.0]
    out, lse = C.lse_combine(O, lse2)
    assert np.array_equal(out, O[2])
    assert np.allclose(lse, lse2[2] * np.log(2.0), rtol=0, atol=1e-15)


def test_equal_lses_give_the_mean():
    rng = np.random.default_rng(2)
    S = 8
    O = rng.standard_normal((S, 5, 16))
    lse2 = np.full((S, 5), 7.25)
    out, lse = C.lse_combine(O, lse2)
    assert np.allclose(out, O.mean(axis=0), rtol=0, atol=1e-14)
    assert np.allclose(lse, 7.25 * np.log(2.0) + np.log(S), rtol=0, atol=1e-13)


def test_all_empty_gives_zero_and_neg_inf():
    O = np.full((3, 2, 4), 7.0)
    lse2 = np.full((3, 2), -np.inf)
    out, lse = C.lse_combine(O, lse2)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_base_two_is_converted():
    # One shard with base-2 LSE 1: the natural-log LSE is ln 2, not 1.
    out, lse = C.lse_combine(np.ones((1, 1, 1)), np.array([[1.0]]))
    assert abs(lse[0] - np.log(2.0)) < 1e-15
    # Two shards with base-2 LSE 0 and 1 weigh 1:2.
    O = np.array([[[0.0]], [[3.0]]])
    out, lse = C.lse_combine(O, np.array([[0.0], [1.0]]))
    assert abs(out[0, 0] - 2.0) < 1e-15
    assert abs(lse[0] - np.log(3.0)) < 1e-15


def test_bf16_decode_is_exact():
    import torch
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(C.bf16_to_f64(bits), x.to(torch.float64).numpy())
