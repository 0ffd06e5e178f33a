"""dsa_indexer_steps_noalloc: the step kernels with the candidate buffer in the
library's static device array.  Host-side argument checks on the CPU; on the
GPU, two calls in a row (the second reusing the array) against the same entry
points run with a caller-owned candidate buffer, bit for bit."""
import ctypes

import numpy as np
import pytest

from dsa_sparse_indexer_gb300 import _lib

OK, INVALID, UNSUPPORTED = 0, 1, 2
NULL = None
SCRATCH = 64 << 20


@pytest.fixture(scope="module")
def lib():
    from dsa_sparse_indexer_gb300 import build as B
    B.build()
    return _lib.load()


def test_host_checks(lib):
    f = lib.dsa_indexer_steps_noalloc
    args = lambda rows, S, K: (NULL, 64, rows, S, 1, K, NULL, NULL, NULL, 1, 1, 64, NULL, NULL,
                               NULL, NULL, NULL, NULL)
    assert f(*args(0, 4, 2048)) == OK                       # nothing to do
    assert f(*args(-1, 4, 2048)) == INVALID
    rows = SCRATCH // (4 * 2048 * 8) + 1                    # one row past the array
    assert f(*args(rows, 4, 2048)) == UNSUPPORTED


# Fake, 16-byte-aligned device addresses: every case below fails a host check
# before anything is enqueued, so none of them is ever dereferenced.
_PTR = 1 << 20


def _full_args(rows=4, S=4, I=1, K=2048, ld=64, bt=_PTR, reqs=1, max_blocks=1, block_size=64,
               ids=_PTR, slots=_PTR, row_ends=_PTR, logits=_PTR):
    return (logits, ld, rows, S, I, K, NULL, row_ends, bt, reqs, max_blocks, block_size, NULL,
            ids, slots, NULL, NULL, NULL)


@pytest.mark.parametrize("rows", [0, 4])
@pytest.mark.parametrize("bad, want", [
    (dict(block_size=0), INVALID), (dict(reqs=0), INVALID), (dict(max_blocks=0), INVALID),
    (dict(I=0), UNSUPPORTED), (dict(ld=6), INVALID), (dict(ld=0), INVALID),
    (dict(S=65), UNSUPPORTED), (dict(K=777), UNSUPPORTED)])
def test_scalar_checks_of_every_step_come_first(lib, rows, bad, want):
    """A bad scalar of any of the three steps (the convert's block size, the
    local top-K's stride, ...) is reported whether or not there are rows."""
    assert lib.dsa_indexer_steps_noalloc(*_full_args(rows=rows, **bad)) == want


@pytest.mark.parametrize("bad", [dict(bt=NULL), dict(ids=NULL), dict(slots=NULL),
                                 dict(row_ends=NULL), dict(logits=NULL), dict(logits=_PTR + 4)])
def test_a_later_steps_pointer_check_runs_before_any_launch(lib, bad):
    """With rows > 0, a null block table, ids or slots (checked by the merge
    and the convert) is reported before the local top-K is queued; these
    calls never reach the GPU (there is none here)."""
    assert lib.dsa_indexer_steps_noalloc(*_full_args(**bad)) == INVALID


@pytest.mark.gpu
def test_two_calls_match_the_entry_points_with_a_caller_buffer(lib):
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    from tests import gpu_cases as G
    from tests.test_gpu_parity import _ties_and_tails_case

    for case in (G.make_case("tiny"), _ties_and_tails_case(1024, 4, 3, rows=24)):
        cfg = case["cfg"]
        logits, starts, ends = G.dev(case["local"]), G.dev(case["starts"]), G.dev(case["ends"])
        bt = G.dev(case["bt"])
        want = G.run_gpu(case)
        assert want["err"] == 0
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        for _ in range(2):
            ids = torch.full((cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
            slots = torch.full((cfg.S, cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
            counts = torch.full((cfg.S, cfg.rows), 7, dtype=torch.int32, device="cuda")
            err = dsa.new_error_flags("cuda")
            st = lib.dsa_indexer_steps_noalloc(
                P(logits), cfg.ld, cfg.rows, cfg.S, cfg.I, cfg.K, P(starts), P(ends), P(bt),
                cfg.reqs, cfg.max_blocks, cfg.block_size, None, P(ids), P(slots), P(counts),
                P(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
            assert st == OK
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            np.testing.assert_array_equal(ids.cpu().numpy(), want["ids"])
            np.testing.assert_array_equal(slots.cpu().numpy(), want["slots"])
            np.testing.assert_array_equal(counts.cpu().numpy(), want["counts"])

        # A bad argument of the last step (a zero block size) is found before
        # the first kernel: the ids, slots and counts keep their fill.
        ids = torch.full((cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
        slots = torch.full((cfg.S, cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
        counts = torch.full((cfg.S, cfg.rows), 7, dtype=torch.int32, device="cuda")
        st = lib.dsa_indexer_steps_noalloc(
            P(logits), cfg.ld, cfg.rows, cfg.S, cfg.I, cfg.K, P(starts), P(ends), P(bt),
            cfg.reqs, cfg.max_blocks, 0, None, P(ids), P(slots), P(counts), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == INVALID
        torch.cuda.synchronize()
        assert (ids == 7).all() and (slots == 7).all() and (counts == 7).all()
