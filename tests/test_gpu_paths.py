"""GPU parity of the throughput kernels' fallback paths on crafted rows.

Every merge row runs twice: alone (a batch that fits one wave takes the
latency kernel: all candidates in registers, one histogram linear in the
score over their range) and tiled to 400 rows (the throughput kernel).  The
throughput merge sets a floor from candidates at fixed sample positions; these
rows make the estimate miss in each way it handles: the floor lands
above the K-th key (every valid candidate is taken again), too many keys sit
at or above it (the list overflows into the radix path), no floor is needed
at all, and the threshold bin is crowded with ties.  The throughput local
top-K bins the keys linearly in the score over their range; its rows hold an
infinite score, an outlier that puts nearly every key into one bin, coarse
ties, and a block of high scores.  Each result is compared element by element
with the oracle.
"""
import numpy as np
import pytest

from oracle import indexer as OX

pytestmark = pytest.mark.gpu


# Batches that fit one wave take the latency kernel (all candidates in
# registers); larger ones the throughput kernel (sampled floor and list).
ROWS_LATENCY, ROWS_THROUGHPUT = 1, 400


def _merge_check(scores: np.ndarray, ids: np.ndarray, K: int) -> None:
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    cand = np.stack([scores.astype(np.float32), ids.astype(np.int32).view(np.float32)], -1)
    want_ids, want_sc = OX.merge(scores, ids, K)
    for rows in (ROWS_LATENCY, ROWS_THROUGHPUT):
        t = torch.from_numpy(np.tile(cand[None], (rows, 1, 1)))
        err = dsa.new_error_flags("cuda")
        got_ids, got_sc = dsa.merge_topk_stable(t.cuda(), K, want_scores=True, err_flags=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got_ids, got_sc = got_ids.cpu().numpy(), got_sc.cpu().numpy()
        for r in (0, rows - 1):
            np.testing.assert_array_equal(got_ids[r], want_ids)
            np.testing.assert_array_equal(got_sc[r], want_sc)


def _merge_sampled(C: int, nt: int = 256) -> np.ndarray:
    """Candidates the throughput merge samples in a row of C <= 32 nt candidates:
    candidate i % 2 of float4 (5 i) nt + t of the row, for i < 4, t < nt."""
    t = np.arange(nt)
    pos = np.concatenate([2 * ((5 * i) * nt + t) + (i & 1) for i in range(4)])
    return np.sort(pos[pos < C])


def _unique_ids(rng, n: int) -> np.ndarray:
    return rng.permutation(10 * n)[:n].astype(np.int64)


def test_merge_floor_above_the_kth_key_retries():
    """Sampled candidates score high, the rest low: the sample floor is above
    the K-th key, so the merge takes every valid candidate (fewer than its list
    holds) and ranks them."""
    rng = np.random.default_rng(1)
    C, K, valid = 4096, 2048, 2900
    scores = rng.standard_normal(C).astype(np.float32)
    samp = _merge_sampled(C)
    scores[samp] = 100.0 + np.arange(len(samp), dtype=np.float32) / 8
    ids = _unique_ids(rng, C)
    ids[valid:] = -1
    scores[valid:] = -np.inf
    _merge_check(scores, ids, K)


def test_merge_list_overflow_takes_the_radix_path():
    """5000 equal candidates at the sampled quantile: more keys at or above the
    floor than the list holds, and ties broken by id."""
    rng = np.random.default_rng(2)
    C, K = 8192, 2048
    scores = rng.standard_normal(C).astype(np.float32)
    scores[rng.permutation(C)[:5000]] = 0.5
    _merge_check(scores, _unique_ids(rng, C), K)


def test_merge_without_a_floor():
    """Fewer valid candidates than 1.25 K: no sample floor; every valid one is
    ranked (padding interleaved with the candidates)."""
    rng = np.random.default_rng(3)
    C, K = 8192, 2048
    scores = rng.standard_normal(C).astype(np.float32)
    ids = _unique_ids(rng, C)
    pad = rng.permutation(C)[:C - 2300]
    ids[pad] = -1
    scores[pad] = -np.inf
    _merge_check(scores, ids, K)


@pytest.mark.parametrize("K", [512, 2048])
def test_merge_crowded_threshold_bin(K):
    """Scores on a coarse grid: bins around the K-th key hold many ties."""
    rng = np.random.default_rng(4 + K)
    C = 4 * K
    scores = (np.rint(rng.standard_normal(C) * 2) / 2).astype(np.float32)
    _merge_check(scores, _unique_ids(rng, C), K)


@pytest.mark.parametrize("special", [np.inf, -np.inf])
def test_merge_infinite_scores(special):
    """Valid candidates scoring +-inf: no finite range to bin, so the latency
    kernel takes the exact radix path; the throughput kernel's floor handles them."""
    rng = np.random.default_rng(9)
    C, K = 8192, 2048
    scores = rng.standard_normal(C).astype(np.float32)
    scores[[3, 4000, 8000]] = special
    _merge_check(scores, _unique_ids(rng, C), K)


def test_merge_an_outlier_crowds_one_bin():
    """One candidate at 1e30: every other key falls into the lowest bin of a
    range-wide histogram."""
    rng = np.random.default_rng(10)
    C, K = 8192, 512
    scores = rng.standard_normal(C).astype(np.float32)
    scores[77] = 1e30
    _merge_check(scores, _unique_ids(rng, C), K)


def _topk_check(row: np.ndarray, n: int, K: int) -> None:
    """One shard (S = 1, I = 1), one row with local range [0, n)."""
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    ld = (len(row) + 3) // 4 * 4
    logits = np.full((1, 1, ld), np.nan, np.float32)
    logits[0, 0, :len(row)] = row
    ends = torch.tensor([n], dtype=torch.int32, device="cuda")
    err = dsa.new_error_flags("cuda")
    local_idx = dsa.shard_topk(torch.from_numpy(logits).cuda(), ends, K, 1, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(local_idx.cpu().numpy()[0, 0], OX.shard_topk(row, 0, n, K))


def test_local_topk_a_block_of_high_scores():
    """A quarter of the slots (a regular pattern over the register layout)
    score far above the rest: the K-th key lies in the bulk, far below the
    block, and the bins between them stay empty."""
    rng = np.random.default_rng(5)
    n, K = 7000, 2048
    row = rng.standard_normal(8192).astype(np.float32)
    t = np.arange(512)
    samp = np.concatenate([4 * (512 * i + t) + i for i in range(4)])
    samp = samp[samp < n]
    row[samp] = 50.0 + np.arange(len(samp), dtype=np.float32) / 64
    _topk_check(row, n, K)


def test_local_topk_crowded_threshold_bin():
    """Coarse-grid values: the bin of the K-th key holds more keys than the
    ranking handles, so the radix select takes over (ties by slot)."""
    rng = np.random.default_rng(6)
    n, K = 8000, 1024
    row = (np.rint(rng.standard_normal(8192) * 2) / 2).astype(np.float32)
    _topk_check(row, n, K)


@pytest.mark.parametrize("special", [np.inf, -np.inf])
def test_local_topk_infinite_scores_take_the_radix_select(special):
    """An infinite score leaves no finite score range to bin: the radix select
    over the registers takes over (the infinite key still ranks by value)."""
    rng = np.random.default_rng(7)
    n, K = 7000, 2048
    row = rng.standard_normal(8192).astype(np.float32)
    row[[5, 4000]] = special
    _topk_check(row, n, K)


def test_local_topk_an_outlier_crowds_one_bin():
    """One score of 1e30: every other key falls into the lowest bin, far more
    than the ranking handles, so the radix select takes over."""
    rng = np.random.default_rng(8)
    n, K = 8000, 512
    row = rng.standard_normal(8192).astype(np.float32)
    row[123] = 1e30
    _topk_check(row, n, K)


@pytest.mark.parametrize("spread", [1e-4, 1e-3, 1e-2])
def test_local_topk_scores_far_from_zero(spread):
    """Scores 100 + N(0,1) * spread: the narrower the range next to the scores'
    size, the coarser the FFMA bin map's offset (at 1e-4 it is off by several
    bins, and the end check sends the row to the radix select; at 1e-2 the map
    holds).  Whichever path the end check picks, the selection is exact."""
    rng = np.random.default_rng(11)
    n, K = 8100, 2048
    row = (100.0 + rng.standard_normal(8192) * spread).astype(np.float32)
    _topk_check(row, n, K)


def test_local_topk_signed_zeros_at_the_threshold_keep_their_sign():
    """The K-th score is a zero shared by 30 slots (-0.0 and +0.0 alternating,
    equal as scores): the first 8 of them by slot win, and each packed
    candidate carries its own zero's sign bit."""
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    rng = np.random.default_rng(12)
    n, K = 8192, 2048
    row = -1.0 - rng.random(n).astype(np.float32)             # the bulk, below -1
    hi = rng.permutation(n)[:2040 + 30]
    row[hi[:2040]] = 1.0 + rng.random(2040).astype(np.float32)  # 2040 clear winners
    zeros = np.sort(hi[2040:])
    row[zeros] = np.where(np.arange(30) % 2 == 0, -0.0, 0.0).astype(np.float32)
    _topk_check(row, n, K)

    logits = torch.from_numpy(row.reshape(1, 1, n)).cuda()
    ends = torch.tensor([n], dtype=torch.int32, device="cuda")
    err = dsa.new_error_flags("cuda")
    local_idx, cand = dsa.shard_topk_pack(logits, ends, K, 1, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    li = local_idx.cpu().numpy()[0, 0]
    np.testing.assert_array_equal(li, OX.shard_topk(row, 0, n, K))
    got = cand.cpu().numpy()[0, :, 0]
    np.testing.assert_array_equal(got.view(np.uint32), row[li].view(np.uint32))
    assert np.array_equal(np.intersect1d(li, zeros), zeros[:8])


@pytest.mark.parametrize("ld,K", [(8192, 2048), (8196, 2048), (16384, 2048), (8196, 512)])
def test_local_topk_at_the_kernel_size_boundaries(ld, K):
    """Rows whose allocated length sits at or just past a kernel variant's
    capacity (256 threads x 32 scores up to 8192 slots, 512 x 32 up to
    16384): ranges ending at ld, ranges just above K with an unaligned start
    (the copy starts at the float4 holding it), a range one slot short of ld.
    Bit-exact against the oracle (S = 1, I = 1: local slots are the row's)."""
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    rng = np.random.default_rng(ld + K)
    ranges = [(0, ld), (3, K + 4), (7, ld - 1)]
    rows = len(ranges)
    x = rng.standard_normal((1, rows, ld)).astype(np.float32)
    starts = torch.tensor([a for a, _ in ranges], dtype=torch.int32, device="cuda")
    ends = torch.tensor([b for _, b in ranges], dtype=torch.int32, device="cuda")
    err = dsa.new_error_flags("cuda")
    local_idx = dsa.shard_topk(torch.from_numpy(x).cuda(), ends, K, 1, row_starts=starts,
                               err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = local_idx.cpu().numpy()[0]
    for r, (lo, hi) in enumerate(ranges):
        np.testing.assert_array_equal(got[r], OX.shard_topk(x[0, r], lo, hi, K))
