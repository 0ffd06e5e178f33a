"""DSA_FLAG_TIMEOUT: a bounded mbarrier wait that runs out, on the GPU, with
no fault and no hang.

A separate test-only library (`build_stalled_copy_test`: shard_topk.cu built
with DSA_TEST_STALLED_COPY, never libdsa.so) adds one mbarrier to the staging
wait of the local top-K, armed for 16 bytes that no copy delivers, and cuts
the poll bound to 4096.  Every real bulk copy still lands (its own barrier
completes); the extra wait runs out, the kernel raises DSA_FLAG_TIMEOUT in the
caller's error word, drains its copies and returns without writing its
outputs.  The same context then runs the production library to full parity.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from oracle import dcp_layout as OL
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu

FLAG_BOUNDS, FLAG_TIMEOUT = 1, 2


@pytest.fixture(scope="module")
def stalled_lib():
    from dsa_sparse_indexer_gb300 import build as B
    lib = ctypes.CDLL(B.build_stalled_copy_test())
    p, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.dsa_shard_topk.argtypes = [p, i64, i, i, i, i, p, p, p, p, p]
    lib.dsa_shard_topk.restype = i
    return lib


def _staged_case():
    """Local rows of 20-24 K slots (above the register path's 16384, inside the
    staging capacity): the local top-K stages them with bulk copies."""
    rng = np.random.default_rng(21)
    rows, S, I, K, ld = 2, 1, 1, 2048, 24000
    x = rng.standard_normal((rows, ld)).astype(np.float32)
    ends = np.array([ld, ld - 4001], np.int32)
    cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=64, max_len=ld, ld=ld,
                   reqs=rows, max_blocks=(ld + 63) // 64)
    local = OL.shard_rows(x, ends, S, I, ld)
    bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)])
    return dict(cfg=cfg, x=x, local=local, starts=np.zeros(rows, np.int32), ends=ends, bt=bt,
                r2q=None)


def test_a_stalled_copy_sets_the_timeout_flag_and_the_device_stays_usable(stalled_lib):
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    case = _staged_case()
    cfg = case["cfg"]
    logits, ends = G.dev(case["local"]), G.dev(case["ends"])
    out = torch.full((cfg.S, cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
    err = dsa.new_error_flags("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):          # the second call starts from a clean barrier too
        err.zero_()
        st = stalled_lib.dsa_shard_topk(logits.data_ptr(), cfg.ld, cfg.rows, cfg.S, cfg.I, cfg.K,
                                        None, ends.data_ptr(), out.data_ptr(), err.data_ptr(),
                                        stream)
        assert st == 0
        torch.cuda.synchronize()             # returns: no hang, no fault
        assert int(err.item()) & FLAG_TIMEOUT
        assert not int(err.item()) & FLAG_BOUNDS
        assert (out == 7).all()              # a timed-out CTA writes nothing

    # The context is intact: the production library runs the same rows to parity.
    got = G.run_gpu(case)
    assert got["err"] == 0
    G.assert_indexer_parity(case, got, np.arange(cfg.rows))
