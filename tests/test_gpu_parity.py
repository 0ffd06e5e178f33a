"""CUDA path vs the oracle, element by element, on all five workloads at full
size (sampled rows where the oracle would be slow), plus edge cases.

Indices and packed candidates must match bit for bit; combined outputs within
the tolerance written in gpu_cases.combine_tolerance.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import dcp_layout as OL
from oracle import pipeline as OP
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu


def sample_rows(cfg, n, seed=0):
    if cfg.rows <= n:
        return np.arange(cfg.rows)
    rng = np.random.default_rng(seed)
    pick = rng.choice(np.arange(1, cfg.rows - 1), n - 2, replace=False)
    return np.sort(np.concatenate([[0, cfg.rows - 1], pick]))


@pytest.mark.parametrize("name,nsample", [("tiny", 4), ("decode", 64), ("long_decode", 128),
                                          ("prefill", 40), ("ragged", 256)])
def test_indexer_parity_full_size(name, nsample):
    case = G.make_case(name)
    got = G.run_gpu(case, fused=True)
    G.assert_indexer_parity(case, got, sample_rows(case["cfg"], nsample))
    if case["cfg"].rows > nsample:
        # every row, over host processes (the sampled rows above also checked
        # the merged ids against a brute-force sort of the unsharded row)
        assert G.assert_all_rows_match_oracle(name, got) == case["cfg"].rows


@pytest.mark.parametrize("name", ["tiny", "ragged", "long_decode"])
def test_unfused_path_matches_fused(name):
    case = G.make_case(name)
    a = G.run_gpu(case, fused=True)
    b = G.run_gpu(case, fused=False)
    for k in ("local_idx", "cand_ids", "ids", "slots", "counts"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(G.bits(a["cand_scores"]), G.bits(b["cand_scores"]))
    assert a["err"] == b["err"] == 0


def test_merge_alone_on_oracle_candidates():
    """The merge kernel fed the oracle's own packed candidates."""
    import dsa_sparse_indexer_gb300 as dsa
    case = G.make_case("long_decode")
    cfg = case["cfg"]
    rows = np.arange(0, cfg.rows, 5)
    want = G.run_oracle(case, rows)
    cand = np.stack([want["cand_scores"], want["cand_ids"].astype(np.int32).view(np.float32)],
                    axis=-1)
    ids, scores = dsa.merge_topk_stable(G.dev(cand), cfg.K, want_scores=True)
    np.testing.assert_array_equal(ids.cpu().numpy(), want["ids"])
    np.testing.assert_array_equal(scores.cpu().numpy(), want["scores"])


@pytest.mark.parametrize("name,nsample", [("tiny", 4), ("decode", 64), ("long_decode", 128),
                                          ("prefill", 40), ("ragged", 256)])
def test_fused_cluster_kernel_parity_full_size(name, nsample):
    case = G.make_case(name)
    got = G.run_gpu_fused(case)
    G.assert_indexer_parity(case, got, sample_rows(case["cfg"], nsample))
    if case["cfg"].rows > nsample:
        assert G.assert_all_rows_match_oracle(name, got) == case["cfg"].rows
    lean = G.run_gpu_fused(case, with_intermediates=False)   # the benchmark's call
    for k in ("ids", "slots", "counts"):
        np.testing.assert_array_equal(lean[k], got[k])


def test_reads_stay_inside_each_rows_range():
    """+inf canaries at every slot past a row's end must never be selected."""
    case = G.make_case("ragged", fill=np.inf)
    got = G.run_gpu(case)
    G.assert_indexer_parity(case, got, sample_rows(case["cfg"], 48, seed=3))
    assert np.all(np.isfinite(got["cand_scores"]) | np.isneginf(got["cand_scores"]))


def _ties_and_tails_case(K, S, I, rows=24):
    """Many ties (coarse grid with -0.0), ragged ends around K, I*S and tile
    sizes, a row of equal scores, a row of -inf, a few nonzero starts."""
    rng = np.random.default_rng(K + 10 * S + I)
    Lmax = 3 * K * S + 37
    x = (np.rint(rng.standard_normal((rows, Lmax)) * 4) / 4).astype(np.float32)
    x[rng.random((rows, Lmax)) < 0.05] = -0.0
    x[3] = 0.0                                     # a row of equal scores
    x[4] = -np.inf                                 # a row of -inf (still selectable)
    ends = rng.integers(0, Lmax + 1, rows).astype(np.int32)
    ends[:6] = [Lmax, Lmax, K - 1, Lmax, Lmax, I * S - 1]
    ends[6:9] = [K * S, K * S + 1, 0]
    starts = np.zeros(rows, np.int32)
    starts[10:14] = rng.integers(0, 50, 4)
    ends[10:14] = np.maximum(ends[10:14], starts[10:14])
    ld = (max(OL.local_count(Lmax, s, S, I) for s in range(S)) + 3) // 4 * 4
    cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=16, max_len=Lmax, ld=ld,
                   reqs=rows, max_blocks=(ld + 15) // 16)
    local = OL.shard_rows(x, ends, S, I, ld, fill=np.nan)
    bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)
                   for _ in range(S)])
    return dict(cfg=cfg, x=x, local=local, starts=starts, ends=ends, bt=bt, r2q=None)


@pytest.mark.parametrize("K", [512, 1024, 2048])
@pytest.mark.parametrize("S,I", [(1, 1), (3, 2), (8, 1), (5, 7)])
def test_small_shapes_ties_and_tails(K, S, I):
    """Ties and tails through the step kernels (both packings) and the fused kernel."""
    case = _ties_and_tails_case(K, S, I)
    rows = case["cfg"].rows
    for fused in (True, False):
        got = G.run_gpu(case, fused=fused)
        G.assert_indexer_parity(case, got, np.arange(rows))
    G.assert_indexer_parity(case, G.run_gpu_fused(case), np.arange(rows))


@pytest.mark.parametrize("K", [512, 2048])
@pytest.mark.parametrize("S,I", [(16, 3), (12, 1)])
def test_many_shards_step_kernels(K, S, I):
    """More shards than the fused kernel's cluster holds (S > 8): the step
    kernels alone, including the general convert and the widest merge."""
    case = _ties_and_tails_case(K, S, I, rows=16)
    got = G.run_gpu(case, fused=True)
    G.assert_indexer_parity(case, got, np.arange(case["cfg"].rows))


@pytest.mark.parametrize("K,S,I", [(2048, 64, 1), (1024, 40, 3)])
def test_widest_rows_take_the_wide_merge(K, S, I):
    """More than 32768 candidates a row, up to the largest shard count: the
    merge's select-and-sort kernel for wide rows (ties on a coarse grid, so
    its second select on the ids runs too), through the step kernels."""
    case = _ties_and_tails_case(K, S, I, rows=16)
    got = G.run_gpu(case, fused=True)
    G.assert_indexer_parity(case, got, np.arange(case["cfg"].rows))


@pytest.mark.parametrize("ld", [24000, 60000])
def test_rows_longer_than_the_register_path(ld):
    """Local rows above the register capacity (16384) are staged in shared
    memory (ld 24000) or, above the staging capacity, read from global memory
    (ld 60000); with S=16 the merge's candidates exceed shared memory too."""
    rng = np.random.default_rng(11)
    rows, S, I, K = 3, 16, 1, 2048
    Lmax = 16 * ld
    x = rng.standard_normal((rows, Lmax)).astype(np.float32)
    ends = np.array([Lmax, Lmax - 1001, 5000], np.int32)
    cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=64, max_len=Lmax, ld=ld,
                   reqs=rows, max_blocks=(ld + 63) // 64)
    local = OL.shard_rows(x, ends, S, I, ld)
    bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)
                   for _ in range(S)])
    case = dict(cfg=cfg, x=x, local=local, starts=np.zeros(rows, np.int32), ends=ends, bt=bt,
                r2q=None)
    got = G.run_gpu(case)
    G.assert_indexer_parity(case, got, np.arange(rows))


def test_very_long_local_rows():
    """Quarter-million-slot local rows (2 shards, 512 K tokens a row): the
    global-memory select over many radix passes, K = 512 and 2048."""
    rng = np.random.default_rng(13)
    for K in (512, 2048):
        rows, S, I = 2, 2, 3
        Lmax = 2 * 262144
        ld = (max(OL.local_count(Lmax, s, S, I) for s in range(S)) + 3) // 4 * 4
        x = rng.standard_normal((rows, Lmax)).astype(np.float32)
        ends = np.array([Lmax, Lmax - 77777], np.int32)
        cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=64, max_len=Lmax,
                       ld=ld, reqs=rows, max_blocks=(ld + 63) // 64)
        local = OL.shard_rows(x, ends, S, I, ld)
        bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)
                       for _ in range(S)])
        case = dict(cfg=cfg, x=x, local=local, starts=np.zeros(rows, np.int32), ends=ends,
                    bt=bt, r2q=None)
        G.assert_indexer_parity(case, G.run_gpu(case), np.arange(rows))
        G.assert_indexer_parity(case, G.run_gpu_fused(case), np.arange(rows))


@pytest.mark.parametrize("ld", [30000, 52000])
def test_fused_rows_longer_than_the_register_path(ld):
    """The fused kernel's staged (ld 30000) and global-memory (ld 52000) paths."""
    rng = np.random.default_rng(12)
    rows, S, I, K = 3, 8, 2, 1024
    Lmax = S * ld
    x = (np.rint(rng.standard_normal((rows, Lmax)) * 16) / 16).astype(np.float32)
    ends = np.array([Lmax, Lmax - 999, 3000], np.int32)
    cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=32, max_len=Lmax, ld=ld,
                   reqs=rows, max_blocks=(ld + 31) // 32)
    local = OL.shard_rows(x, ends, S, I, ld)
    bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)
                   for _ in range(S)])
    case = dict(cfg=cfg, x=x, local=local, starts=np.zeros(rows, np.int32), ends=ends, bt=bt,
                r2q=None)
    G.assert_indexer_parity(case, G.run_gpu_fused(case), np.arange(rows))


def test_out_of_range_ends_and_tables_set_the_bounds_flag():
    import dsa_sparse_indexer_gb300 as dsa
    S, I, K, rows, ld = 2, 1, 512, 2, 1024
    logits = torch.randn(S, rows, ld, device="cuda")
    ends = torch.tensor([2 * ld + 8, 100], dtype=torch.int32, device="cuda")  # row 0 too long
    err = dsa.new_error_flags("cuda")
    idx = dsa.shard_topk(logits, ends, K, I, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dsa.DSA_FLAG_BOUNDS
    # the clipped row still selects from [0, ld) only
    assert int(idx.max()) < ld
    # a block table too narrow for the ids
    ids = torch.arange(K, dtype=torch.int32, device="cuda").repeat(rows, 1)
    bt = torch.zeros(S, rows, 2, dtype=torch.int32, device="cuda")   # 2 blocks of 16
    err.zero_()
    slots, counts = dsa.convert_index_compact(ids, bt, 16, I, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dsa.DSA_FLAG_BOUNDS
    assert counts.cpu().numpy().tolist() == [[K // 2] * rows] * S
    s = slots.cpu().numpy()
    assert np.all(s[:, :, :32] >= 0) and np.all(s[:, :, 32:] == -1)


def test_zero_rows_is_a_no_op():
    import dsa_sparse_indexer_gb300 as dsa
    logits = torch.zeros(2, 0, 64, device="cuda")
    out = dsa.shard_topk(logits, torch.zeros(0, dtype=torch.int32, device="cuda"), 512, 1)
    assert out.shape == (2, 0, 512)
    o = dsa.indexer_fused(logits, torch.zeros(0, dtype=torch.int32, device="cuda"), 512, 1,
                          torch.zeros(2, 1, 4, dtype=torch.int32, device="cuda"), 64)
    assert o["ids"].shape == (0, 512)


def _combine_case(name, rows=None):
    cfg = W.CONFIGS[name]
    case = G.make_case(name)
    R = cfg.rows if rows is None else rows
    want = G.run_oracle(case, np.arange(R))
    empty = want["counts"] == 0                   # shards with no selected token
    part, lse2 = W.combine_inputs(cfg, empty=empty, rows=R)
    return cfg, part, lse2, empty


@pytest.mark.parametrize("name", ["ragged", "decode"])
def test_lse_combine_parity_full_size(name):
    import dsa_sparse_indexer_gb300 as dsa
    cfg, part, lse2, empty = _combine_case(name)
    if name == "ragged":
        assert empty.any() and (~empty).any()
    g = G.Guards()
    R, H, D = cfg.rows, cfg.H, cfg.D
    out, lse = dsa.lse_combine(G.dev(part.view(np.int16)).view(torch.bfloat16), G.dev(lse2),
                               out=g.empty((R, H, D), torch.bfloat16),
                               lse_out=g.empty((R, H), torch.float32))
    g.check()
    # every row, 32 at a time (the fp64 oracle holds S x 32 x H x D values)
    for c in np.array_split(np.arange(cfg.rows), max(1, cfg.rows // 32)):
        G.assert_combine_parity(out, lse, part, lse2, c)


@pytest.mark.parametrize("S,H,D", [(1, 3, 8), (8, 5, 136), (3, 2, 520), (40, 2, 64),
                                   (64, 1, 256), (4, 2, 2304), (2, 2, 4096), (7, 2, 1024)])
def test_lse_combine_shapes_and_degenerate_cases(S, H, D):
    import dsa_sparse_indexer_gb300 as dsa
    rng = np.random.default_rng(S * 7 + D)
    rows = 9
    part = W.f32_to_bf16_bits(rng.standard_normal((S, rows, H, D)).astype(np.float32))
    lse2 = rng.uniform(-5, 20, (S, rows, H)).astype(np.float32)
    lse2[:, 0] = -np.inf                     # every shard empty -> 0, -inf
    lse2[1:, 1] = -np.inf                    # one shard only
    lse2[:, 2] = 3.5                         # equal LSEs -> mean
    lse2[0, 3] = 60.0                        # one shard dominates
    part[:, 0] = 0
    g = G.Guards()
    out, lse = dsa.lse_combine(G.dev(part.view(np.int16)).view(torch.bfloat16), G.dev(lse2),
                               out=g.empty((rows, H, D), torch.bfloat16),
                               lse_out=g.empty((rows, H), torch.float32))
    g.check()
    G.assert_combine_parity(out, lse, part, lse2, np.arange(rows))
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse.cpu().numpy()[0]))


def test_results_do_not_depend_on_the_stream():
    import dsa_sparse_indexer_gb300 as dsa
    case = G.make_case("tiny")
    a = G.run_gpu(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = G.run_gpu(case)
    s.synchronize()
    for k in ("local_idx", "ids", "slots", "counts"):
        np.testing.assert_array_equal(a[k], b[k])
