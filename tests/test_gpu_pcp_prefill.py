"""GPU parity of the PCP prefill cache-row kernels (dsa_fused_norm_rope,
dsa_kv_cache_insert) with the fp64 oracle (oracle/pcp_prefill.py).

Tolerance, from the arithmetic: the kernel computes in fp32 from bf16 inputs
(a 512-term sum of squares, one reciprocal square root, two products per
value; a two-term rotation) and rounds once to bf16.  A bf16 output is then
within half a bf16 ulp of the oracle's unrounded fp64 value plus the fp32
error before that rounding, bounded here by 4e-5 of the value (512 rounded
additions at 2^-24 each, with room) and 1e-6 absolute.  The cache insert is a
copy: bit-exact."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import combine as OC
from oracle import pcp_prefill as PP
from tests import gpu_cases as G

pytestmark = pytest.mark.gpu


def _tol(ref):
    return 0.5 * G.bf16_ulp(ref) + 4e-5 * np.abs(ref) + 1e-6


def _assert_close(got_bits, ref):
    got = OC.bf16_to_f64(got_bits)
    bad = np.abs(got - ref) > _tol(ref)
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _bf(a):
    return G.dev(a.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("T,eps", [(1, 1e-6), (37, 1e-6), (4096, 1e-5)])
def test_materialised_rows_match_the_oracle(T, eps):
    import dsa_sparse_indexer_gb300 as dsa
    kv, kpe, w = W.pcp_token_inputs(T, seed=T)
    table = W.rotation_table(5000, seed=1)
    pos = np.random.default_rng(T).integers(0, 5000, T).astype(np.int32)
    g = G.Guards()
    err = dsa.new_error_flags("cuda")
    kv_out, kpe_out = dsa.fused_norm_rope(_bf(kv), _bf(kpe), G.dev(pos), G.dev(w), eps,
                                          G.dev(table), kv_out=g.empty((T, 512), torch.bfloat16),
                                          kpe_out=g.empty((T, 64), torch.bfloat16), err_flags=err)
    g.check()
    assert int(err.item()) == 0
    ref_kv, ref_kpe = PP.fused_norm_rope(OC.bf16_to_f64(kv), OC.bf16_to_f64(kpe), w, eps, pos,
                                         table)
    _assert_close(_bits(kv_out), ref_kv)
    _assert_close(_bits(kpe_out), ref_kpe)


def test_direct_insert_equals_materialise_then_gather_then_insert():
    """The non-PCP mode (rows straight into the cache) and the PCP mode (rows
    materialised by each rank's slice, gathered, then inserted) fill the cache
    identically, and match the oracle's insert; slots of -1 and the rest of the
    cache are untouched."""
    import dsa_sparse_indexer_gb300 as dsa
    T, P, n_slots = 1000, 4, 3000
    kv, kpe, w = W.pcp_token_inputs(T, seed=5)
    table = W.rotation_table(2048, seed=6)
    rng = np.random.default_rng(7)
    pos = rng.integers(0, 2048, T).astype(np.int32)
    slots = rng.permutation(n_slots)[:T].astype(np.int32)
    slots[::9] = -1
    base = W.f32_to_bf16_bits(rng.standard_normal((n_slots, 576), dtype=np.float32))
    err = dsa.new_error_flags("cuda")

    direct = _bf(base.copy())
    dsa.fused_norm_rope(_bf(kv), _bf(kpe), G.dev(pos), G.dev(w), 1e-6, G.dev(table),
                        materialize=False, slot_mapping=G.dev(slots), kv_cache=direct,
                        err_flags=err)
    # PCP: rank p materialises its contiguous slice into its part of one buffer
    g = G.Guards()
    kv_all, kpe_all = g.empty((T, 512), torch.bfloat16), g.empty((T, 64), torch.bfloat16)
    cuts = np.linspace(0, T, P + 1).astype(int)
    for p in range(P):
        a, b = cuts[p], cuts[p + 1]
        dsa.fused_norm_rope(_bf(kv[a:b]), _bf(kpe[a:b]), G.dev(pos[a:b]), G.dev(w), 1e-6,
                            G.dev(table), kv_out=kv_all[a:b], kpe_out=kpe_all[a:b],
                            err_flags=err)
    pcp = _bf(base.copy())
    dsa.kv_cache_insert(kv_all, kpe_all, G.dev(slots), pcp, err_flags=err)
    g.check()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(_bits(direct), _bits(pcp))
    rows = np.concatenate([_bits(kv_all), _bits(kpe_all)], axis=1)
    np.testing.assert_array_equal(_bits(pcp), PP.cache_insert(base, rows, slots))


def test_bad_positions_and_slots_set_the_bounds_flag():
    import dsa_sparse_indexer_gb300 as dsa
    T = 8
    kv, kpe, w = W.pcp_token_inputs(T, seed=9)
    table = W.rotation_table(100, seed=10)
    pos = np.arange(T, dtype=np.int32)
    pos[3] = 100                                   # past the table: not rotated
    slots = np.arange(T, dtype=np.int32)
    slots[5] = 16                                  # past the cache: skipped
    cache = torch.zeros((16, 576), dtype=torch.bfloat16, device="cuda")
    err = dsa.new_error_flags("cuda")
    kv_out, kpe_out = dsa.fused_norm_rope(_bf(kv), _bf(kpe), G.dev(pos), G.dev(w), 1e-6,
                                          G.dev(table), slot_mapping=G.dev(slots),
                                          kv_cache=cache, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dsa.DSA_FLAG_BOUNDS
    np.testing.assert_array_equal(_bits(kpe_out)[3], kpe[3])
    c = _bits(cache)
    assert (c[5] == 0).all()                       # token 5 went nowhere, slot 5 unused
    np.testing.assert_array_equal(c[4, :512], _bits(kv_out)[4])
