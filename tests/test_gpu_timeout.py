"""DSA_FLAG_TIMEOUT: a bounded mbarrier wait that runs out, on the GPU, with
no fault and no hang.

A separate test-only library (`build_stalled_copy_test`: shard_topk.cu,
attention.cu and indexer_logits.cu built with DSA_TEST_STALLED_COPY, never
libdsa.so) adds one mbarrier, armed for 16 bytes that no copy delivers, to the
staging waits of the local top-K (the staged kernel for long rows and the
shared-memory kernel for rows up to 16384 slots) and before the logits' first
MMA, makes the
attention's stage barriers expect one arrival that nothing makes, and cuts the
poll bound to 4096.  Every real bulk copy still lands (its own barrier
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


def _smem_case():
    """Local rows of 6-8 K slots: the throughput kernel copies each range into
    shared memory with one bulk copy."""
    rng = np.random.default_rng(22)
    rows, S, I, K, ld = 2, 1, 1, 2048, 8000
    x = rng.standard_normal((rows, ld)).astype(np.float32)
    ends = np.array([ld, ld - 1999], np.int32)
    cfg = W.Config("adhoc", 9, rows=rows, S=S, I=I, K=K, block_size=64, max_len=ld, ld=ld,
                   reqs=rows, max_blocks=(ld + 63) // 64)
    local = OL.shard_rows(x, ends, S, I, ld)
    bt = np.stack([rng.permutation(rows * cfg.max_blocks).astype(np.int32).reshape(rows, -1)])
    return dict(cfg=cfg, x=x, local=local, starts=np.zeros(rows, np.int32), ends=ends, bt=bt,
                r2q=None)


def test_a_stalled_copy_in_the_shared_memory_top_k(stalled_lib):
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    case = _smem_case()
    cfg = case["cfg"]
    logits, ends = G.dev(case["local"]), G.dev(case["ends"])
    out = torch.full((cfg.S, cfg.rows, cfg.K), 7, dtype=torch.int32, device="cuda")
    err = dsa.new_error_flags("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        err.zero_()
        st = stalled_lib.dsa_shard_topk(logits.data_ptr(), cfg.ld, cfg.rows, cfg.S, cfg.I, cfg.K,
                                        None, ends.data_ptr(), out.data_ptr(), err.data_ptr(),
                                        stream)
        assert st == 0
        torch.cuda.synchronize()
        assert int(err.item()) & FLAG_TIMEOUT
        assert not int(err.item()) & FLAG_BOUNDS
        assert (out == 7).all()

    got = G.run_gpu(case)
    assert got["err"] == 0
    G.assert_indexer_parity(case, got, np.arange(cfg.rows))


def test_a_stalled_attention_stage_sets_the_timeout_flag_and_the_device_stays_usable(stalled_lib):
    """The tcgen05 sparse MLA decode in the test build: the first tile's stage
    barrier waits for one arrival that never comes.  Every gathered row and the
    query still land; the MMA thread's bounded polling runs out, every role of
    the CTA stops at its next bounded wait, nothing is written, and the tensor
    memory is freed.  The production library then attends the same slots to
    parity."""
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    from oracle import attention as OA
    from oracle import combine as OC
    p, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    stalled_lib.dsa_sparse_mla_decode.argtypes = [p, p, i64, p, p, i, i, i, i, ctypes.c_float,
                                                  p, p, p, p]
    stalled_lib.dsa_sparse_mla_decode.restype = i
    S, R, H, K, n_slots = 2, 3, 128, 512, 5000
    rng = np.random.default_rng(31)
    q = W.mla_query(R, H, seed=32)
    cache = W.mla_cache(S, n_slots, seed=33)
    counts = np.array([[200, 64, 1], [129, 512, 70]])
    slots = rng.integers(0, n_slots, (S, R, K)).astype(np.int32)
    dq = G.dev(q.view(np.int16)).view(torch.bfloat16)
    dc = G.dev(cache.view(np.int16)).view(torch.bfloat16)
    ds, dn = G.dev(slots), G.dev(counts.astype(np.int32))
    out = torch.full((S, R, H, W.MLA_DV), 7, dtype=torch.int16, device="cuda")
    lse2 = torch.full((S, R, H), 7.0, dtype=torch.float32, device="cuda")
    err = dsa.new_error_flags("cuda")
    scale = 1.0 / np.sqrt(192.0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):          # the second call starts from a clean barrier too
        err.zero_()
        st = stalled_lib.dsa_sparse_mla_decode(dq.data_ptr(), dc.data_ptr(), n_slots,
                                               ds.data_ptr(), dn.data_ptr(), R, S, H, K, scale,
                                               out.data_ptr(), lse2.data_ptr(), err.data_ptr(),
                                               stream)
        assert st == 0
        torch.cuda.synchronize()             # returns: no hang, no fault
        assert int(err.item()) & FLAG_TIMEOUT
        assert not int(err.item()) & FLAG_BOUNDS
        assert (out == 7).all() and (lse2 == 7.0).all()   # a timed-out CTA writes nothing

    # The context is intact: the production library attends the same slots.
    o, l2 = dsa.sparse_mla_decode(dq, dc, ds, dn, scale, err_flags=err.zero_())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = OC.bf16_to_f64(o.view(torch.int16).cpu().numpy().view(np.uint16))
    want_o, want_l = OA.shard_attention(OC.bf16_to_f64(q), OC.bf16_to_f64(cache), slots, counts,
                                        scale, W.MLA_DV)
    assert (np.abs(got - want_o) <= G.combine_tolerance(want_o)).all()
    assert (np.abs(l2.cpu().numpy() - want_l) <= 1e-5 * np.maximum(1.0, np.abs(want_l))).all()


def test_a_stalled_logits_mma_sets_the_timeout_flag_and_the_device_stays_usable(stalled_lib):
    """The tcgen05 indexer logits in the test build: before its first MMA the
    issuing thread waits on an mbarrier armed for 16 bytes that no copy
    delivers.  The query and key copies land on their own barriers; the wait
    runs out, the roles stop at their bounded waits, nothing is written, and
    the production library then computes the same logits to parity."""
    import torch

    import dsa_sparse_indexer_gb300 as dsa
    from tests import test_gpu_indexer_logits as TL
    p, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    stalled_lib.dsa_indexer_logits.argtypes = [p, p, p, i64, p, i, i, i, p, p, p, i, i, i, p, i64,
                                               p, p]
    stalled_lib.dsa_indexer_logits.restype = i
    c = TL._case(2, 1, rows=5, Lmax=2 * 1500 + 11, bs=64, seed=51)
    reqs, max_blocks = c["tables"].shape[1], c["tables"].shape[2]
    n_slots = c["k"].shape[1]
    dq, dw, dk = G.dev(c["q"]), G.dev(c["w"]), G.dev(c["k"])
    dt, de, ds0 = G.dev(c["tables"]), G.dev(c["ends"]), G.dev(c["starts"])
    out = torch.full((c["S"], c["rows"], c["ld"]), 7.0, dtype=torch.float32, device="cuda")
    err = dsa.new_error_flags("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):          # the second call starts from a clean barrier too
        err.zero_()
        st = stalled_lib.dsa_indexer_logits(dq.data_ptr(), dw.data_ptr(), dk.data_ptr(), n_slots,
                                            dt.data_ptr(), reqs, max_blocks, c["bs"], None,
                                            ds0.data_ptr(), de.data_ptr(), c["rows"], c["S"],
                                            c["I"], out.data_ptr(), c["ld"], err.data_ptr(),
                                            stream)
        assert st == 0
        torch.cuda.synchronize()             # returns: no hang, no fault
        assert int(err.item()) & FLAG_TIMEOUT
        assert not int(err.item()) & FLAG_BOUNDS
        assert (out == 7.0).all()            # nothing written

    # The context is intact: the production library computes the same logits.
    got, e = TL._run(c)
    assert e == 0
    TL._check(c, got)
