"""GPU parity of the sparse MLA decode attention (dsa_sparse_mla_decode) with
the oracle (oracle/attention.py): first on random slot sets over a seeded
cache (counts from 0 to K, tile tails, H = 64 / 128 / 192), at the decode
batch's full shape in the benchmark's launch configuration (sampled pairs),
then through the whole decode path, the indexer's compacted slots into the
attention and its outputs into the LSE combine, against the oracle pipeline.

Tolerance (derived from the arithmetic): scores are exact bf16 products summed
in fp32, so lse2 is within 1e-5 * max(1, |ref|); the softmax weights enter the
value product rounded to bf16 (relative error 2^-9 each), so an output moves
by at most 2^-9 * max |v - O| (< 8e-3 for the N(0,1) values here) plus its own
bf16 rounding: the combine's bf16 tolerance (1e-2, widened to half an ulp
where an ulp exceeds it)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as OA
from oracle import combine as OC
from oracle import pipeline as OP
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(192.0)


def _attend(q_bits, cache_bits, slots, counts, scale=SCALE):
    import dsa_sparse_indexer_gb300 as dsa
    err = dsa.new_error_flags("cuda")
    g = G.Guards()
    S, rows = counts.shape
    H = q_bits.shape[1]
    out, lse2 = dsa.sparse_mla_decode(G.dev(q_bits.view(np.int16)).view(torch.bfloat16),
                                      G.dev(cache_bits.view(np.int16)).view(torch.bfloat16),
                                      G.dev(slots.astype(np.int32)),
                                      G.dev(counts.astype(np.int32)), scale,
                                      out=g.empty((S, rows, H, W.MLA_DV), torch.bfloat16),
                                      lse2=g.empty((S, rows, H), torch.float32), err_flags=err)
    g.check()
    ob = out.view(torch.int16).cpu().numpy().view(np.uint16)
    return OC.bf16_to_f64(ob), lse2.cpu().numpy(), int(err.item())


def _assert_close(out, lse2, want_out, want_lse2):
    assert np.array_equal(np.isneginf(lse2), np.isneginf(want_lse2))
    fin = np.isfinite(want_lse2)
    assert (np.abs(lse2[fin] - want_lse2[fin]) <= 1e-5 * np.maximum(1.0, np.abs(want_lse2[fin]))).all()
    tol = G.combine_tolerance(want_out)
    bad = np.abs(out - want_out) > tol
    assert not bad.any(), f"{bad.sum()} outputs off; max |d| {np.abs(out - want_out).max()}"


@pytest.mark.parametrize("H", [64, 128, 192])
def test_random_slot_sets(H):
    S, R, K, n_slots = 3, 5, 2048, 9000
    rng = np.random.default_rng(H)
    q = W.mla_query(R, H, seed=10 + H)
    cache = W.mla_cache(S, n_slots, seed=20 + H)
    counts = np.array([[0, 1, 15, 16, 17], [33, 100, 511, 2048, 1],
                       [2047, 64, 0, 1000, 7]])[:S, :R]
    slots = np.full((S, R, K), -1, np.int64)
    for s in range(S):
        for r in range(R):
            slots[s, r, :counts[s, r]] = rng.choice(n_slots, counts[s, r], replace=False)
    out, lse2, err = _attend(q, cache, slots, counts)
    assert err == 0
    want_out, want_lse2 = OA.shard_attention(OC.bf16_to_f64(q), OC.bf16_to_f64(cache), slots,
                                             counts, SCALE, W.MLA_DV)
    _assert_close(out, lse2, want_out, want_lse2)


def test_bad_counts_and_slots_are_flagged_and_left_out():
    S, R, K, H, n_slots = 2, 2, 512, 64, 600
    rng = np.random.default_rng(9)
    q = W.mla_query(R, H, seed=1)
    cache = W.mla_cache(S, n_slots, seed=2)
    slots = rng.integers(0, n_slots, (S, R, K))
    counts = np.array([[40, 7], [3, 0]])
    slots[0, 0, 5] = n_slots + 3                # out of the cache: left out
    slots[1, 0, 1] = -2
    out, lse2, err = _attend(q, cache, slots, counts)
    assert err != 0
    keep = slots.copy()
    cnt = counts.copy()
    for s, r, j in [(0, 0, 5), (1, 0, 1)]:
        row = [x for i, x in enumerate(keep[s, r, :cnt[s, r]]) if i != j]
        cnt[s, r] = len(row)
        keep[s, r, :len(row)] = row
    want_out, want_lse2 = OA.shard_attention(OC.bf16_to_f64(q), OC.bf16_to_f64(cache), keep, cnt,
                                             SCALE, W.MLA_DV)
    _assert_close(out, lse2, want_out, want_lse2)


def _decode_loop(case, H, seed):
    """Indexer (step kernels) -> attention -> combine on the GPU, and the same
    through the oracles."""
    import dsa_sparse_indexer_gb300 as dsa
    cfg = case["cfg"]
    n_slots = cfg.reqs * cfg.max_blocks * cfg.block_size
    q = W.mla_query(cfg.rows, H, seed)
    cache = W.mla_cache(cfg.S, n_slots, seed + 1)
    got = G.run_gpu(case)
    assert got["err"] == 0
    out, lse2, err = _attend(q, cache, got["slots"], got["counts"])
    assert err == 0
    err_t = dsa.new_error_flags("cuda")
    ob = G.dev(W.f32_to_bf16_bits(out.astype(np.float32)).view(np.int16)).view(torch.bfloat16)
    y, lse = dsa.lse_combine(ob, G.dev(lse2.astype(np.float32)), err_flags=err_t)
    torch.cuda.synchronize()
    y = OC.bf16_to_f64(y.view(torch.int16).cpu().numpy().view(np.uint16))
    want = G.run_oracle(case, np.arange(cfg.rows))
    want_out, want_lse2 = OA.shard_attention(OC.bf16_to_f64(q), OC.bf16_to_f64(cache),
                                             want["slots"], want["counts"], SCALE, W.MLA_DV)
    _assert_close(out, lse2, want_out, want_lse2)
    want_y, want_lse = OC.lse_combine(want_out, want_lse2)
    return y, lse.cpu().numpy(), want_y, want_lse


@pytest.mark.parametrize("name,H", [("tiny", 64)])
def test_decode_loop_on_the_tiny_workload(name, H):
    y, lse, want_y, want_lse = _decode_loop(G.make_case(name), H, seed=3)
    # the combined output went through bf16 twice (attention out, combine out)
    assert (np.abs(y - want_y) <= 2 * G.combine_tolerance(want_y)).all()
    fin = np.isfinite(want_lse)
    assert (np.abs(lse[fin] - want_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(want_lse[fin]))).all()


def test_decode_loop_with_ties_and_tails():
    """Ragged rows (empty shards, rows shorter than K, an empty row) at S = 4,
    I = 2, K = 512, H = 64."""
    from tests.test_gpu_parity import _ties_and_tails_case
    y, lse, want_y, want_lse = _decode_loop(_ties_and_tails_case(512, 4, 2), 64, seed=5)
    assert (np.abs(y - want_y) <= 2 * G.combine_tolerance(want_y)).all()
    assert np.array_equal(np.isneginf(lse), np.isneginf(want_lse))
    fin = np.isfinite(want_lse)
    assert (np.abs(lse[fin] - want_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(want_lse[fin]))).all()


def test_decode_batch_size_in_the_benchmarks_launch_configuration():
    """The decode batch's shape as the benchmark launches it (64 rows, S = 4,
    H = 128: 512 CTAs over the SMs, 400-640 selected slots per (row, shard),
    so every CTA runs seven to ten 64-token tiles and some a partial last
    one), caches of 300 K slots per shard (1.4 GB, larger than L2) with the
    benchmark's value distribution; a dozen (row, shard) pairs, the longest
    among them, checked against the oracle."""
    S, R, H, K, n_slots = 4, 64, 128, 2048, 300_000
    rng = np.random.default_rng(77)
    q = W.mla_query(R, H, seed=78)
    cache = W.mla_cache_uniform(S, n_slots, seed=79)
    counts = rng.integers(400, 641, (S, R))
    slots = np.full((S, R, K), -1, np.int64)
    for s in range(S):
        for r in range(R):
            slots[s, r, :counts[s, r]] = rng.integers(0, n_slots, counts[s, r])
    out, lse2, err = _attend(q, cache, slots, counts)
    assert err == 0
    flat = np.argsort(counts, axis=None)
    pairs = [np.unravel_index(i, counts.shape) for i in
             list(flat[-2:]) + list(rng.choice(flat[:-2], 10, replace=False))]
    for s, r in pairs:
        c = counts[s, r]
        want_o, want_l = OA.sparse_mla_decode(OC.bf16_to_f64(q[r]),
                                              OC.bf16_to_f64(cache[s, slots[s, r, :c]]), SCALE,
                                              W.MLA_DV)
        _assert_close(out[s, r], lse2[s, r], want_o, want_l)


@pytest.mark.parametrize("scale", [-1.0 / np.sqrt(192.0), 0.0])
def test_negative_and_zero_scales(scale):
    """The softmax's general path with every token valid: a negative scale
    (the maximum is the most negative dot product) and a zero one (every
    weight 1: O is the plain mean of the selected values, lse2 = log2 n)."""
    S, R, H, K, n_slots = 2, 3, 128, 512, 4000
    rng = np.random.default_rng(41)
    q = W.mla_query(R, H, seed=42)
    cache = W.mla_cache(S, n_slots, seed=43)
    counts = np.array([[64, 300, 1], [512, 65, 128]])
    slots = rng.integers(0, n_slots, (S, R, K))
    out, lse2, err = _attend(q, cache, slots, counts, scale=scale)
    assert err == 0
    want_out, want_lse2 = OA.shard_attention(OC.bf16_to_f64(q), OC.bf16_to_f64(cache), slots,
                                             counts, scale, W.MLA_DV)
    _assert_close(out, lse2, want_out, want_lse2)
    if scale == 0.0:
        np.testing.assert_allclose(lse2, np.log2(counts)[:, :, None] * np.ones(H), rtol=1e-6)
