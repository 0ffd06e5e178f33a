"""The seeded generators: determinism, shapes and recipe properties."""
import numpy as np
import torch

import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -2.0, 0.0, -0.0], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_deterministic_and_shaped():
    cfg = W.CONFIGS["tiny"]
    a = W.global_logits(cfg)
    b = W.global_logits(cfg)
    assert a.shape == (4, 4096) and a.dtype == np.float32
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # 1/64 grid, and the grid produces -0.0
    assert np.all(a * 64 == np.rint(a * 64))
    assert np.any((a == 0) & np.signbit(a))
    assert not np.array_equal(W.global_logits(cfg, replica=1), a)


def test_row_ranges_follow_recipes():
    s, e = W.row_ranges(W.CONFIGS["decode"])
    assert e.min() >= 8192 and e.max() <= 65536 and np.all(s == 0)
    s, e = W.row_ranges(W.CONFIGS["prefill"])
    assert e[0] == 28672 and e[-1] == 28672 + 4095
    s, e = W.row_ranges(W.CONFIGS["ragged"])
    assert e.min() >= 16 and e.max() <= 65536
    assert (e < 1024).any() and (e < 32).any()       # shorter than K and than I*S


def test_long_decode_has_heavy_duplicates():
    cfg = W.CONFIGS["long_decode"]
    x = W.global_logits(cfg)[:2]
    for r in range(2):
        _, counts = np.unique(x[r], return_counts=True)
        dup_frac = 1 - len(counts) / x.shape[1]
        assert 0.07 < dup_frac < 0.13


def test_prefill_mask_beyond_row_end():
    cfg = W.CONFIGS["prefill"]
    _, e = W.row_ranges(cfg)
    x = W.global_logits(cfg)
    for r in (0, 1, 4095):
        assert np.isfinite(x[r, :e[r]]).all() and np.isneginf(x[r, e[r]:]).all()


def test_block_tables_are_permutations():
    cfg = W.CONFIGS["decode"]
    bt = W.block_tables(cfg)
    assert bt.shape == (4, 64, 256)
    for s in range(4):
        assert np.array_equal(np.sort(bt[s].ravel()), np.arange(64 * 256))
    assert not np.array_equal(bt[0], bt[1])
    tiny = W.block_tables(W.CONFIGS["tiny"])
    assert np.array_equal(tiny[1], np.arange(4 * 32).reshape(4, 32))


def test_combine_inputs_respect_empty_mask():
    cfg = W.CONFIGS["ragged"]
    empty = np.zeros((cfg.S, 3), bool)
    empty[2, 1] = True
    out, lse2 = W.combine_inputs(cfg, empty=empty, rows=3)
    assert out.shape == (8, 3, 128, 512) and out.dtype == np.uint16
    assert np.isneginf(lse2[2, 1]).all() and np.all(out[2, 1] == 0)
    ok = ~np.isneginf(lse2)
    assert lse2[ok].min() >= -5 and lse2[ok].max() <= 20


def test_mla_inputs_are_seeded_bf16_of_the_stated_ranges():
    from oracle.combine import bf16_to_f64
    a = W.mla_cache_uniform(2, 300, seed=5)
    b = W.mla_cache_uniform(2, 300, seed=5)
    assert a.shape == (2, 300, W.MLA_DQK) and a.dtype == np.uint16
    assert np.array_equal(a, b)
    v = np.abs(bf16_to_f64(a))
    assert v.min() >= 0.5 and v.max() < 1.0
    q = W.mla_query(3, 64, seed=1)
    assert q.shape == (3, 64, W.MLA_DQK) and np.array_equal(q, W.mla_query(3, 64, seed=1))
    c = bf16_to_f64(W.mla_cache(1, 2000, seed=2))
    assert abs(c.mean()) < 0.01 and abs(c.std() - 1.0) < 0.01
