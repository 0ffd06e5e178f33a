"""The C-ABI library: it loads, exports what include/dsa.h declares, and its host
argument checks reject bad calls before anything reaches a GPU.  No compute."""
import ctypes
import os
import subprocess

import pytest

from dsa_sparse_indexer_gb300 import _lib
from dsa_sparse_indexer_gb300 import build as B

OK, INVALID, UNSUPPORTED = 0, 1, 2
P = 4096            # a fake, 16-byte aligned "device pointer"; never dereferenced
NULL = None


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _lib.declared_functions()
    assert set(declared) == set(_lib.SIGNATURES), declared
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared:
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    assert lib.dsa_version() == 100
    assert _lib.status_string(OK) == "ok"
    assert "invalid" in _lib.status_string(INVALID)
    assert _lib.status_string(99) == "unknown status"


def topk(lib, logits=P, ld=1024, rows=4, S=2, I=1, K=512, starts=NULL, ends=P, out=P):
    return lib.dsa_shard_topk(logits, ld, rows, S, I, K, starts, ends, out, NULL, NULL)


def test_shard_topk_argument_checks(lib):
    assert topk(lib, rows=0) == OK                      # nothing enqueued
    assert topk(lib, logits=NULL) == INVALID
    assert topk(lib, logits=P + 4) == INVALID           # not 16-byte aligned
    assert topk(lib, ld=1022) == INVALID                # ld % 4
    assert topk(lib, ld=0) == INVALID
    assert topk(lib, rows=-1) == INVALID
    assert topk(lib, ends=NULL) == INVALID
    assert topk(lib, out=NULL) == INVALID
    assert topk(lib, S=0) == UNSUPPORTED
    assert topk(lib, S=65) == UNSUPPORTED
    assert topk(lib, I=0) == UNSUPPORTED
    for K in (0, 256, 513, 4096):
        assert topk(lib, K=K) == UNSUPPORTED


def test_pack_and_fused_argument_checks(lib):
    f = lib.dsa_pack_candidates
    assert f(P, 1024, P, 0, 2, 1, 512, P, NULL, NULL) == OK
    assert f(P, 1024, NULL, 4, 2, 1, 512, P, NULL, NULL) == INVALID
    assert f(P, 1024, P, 4, 2, 1, 512, NULL, NULL, NULL) == INVALID
    assert f(P, 1024, P + 8, 4, 2, 1, 512, P, NULL, NULL) == INVALID
    assert f(P, 1024, P, 4, 2, 1, 100, P, NULL, NULL) == UNSUPPORTED
    g = lib.dsa_shard_topk_pack
    assert g(P, 1024, 0, 2, 1, 512, NULL, P, NULL, P, NULL, NULL) == OK
    assert g(P, 1024, 4, 2, 1, 512, NULL, P, NULL, NULL, NULL, NULL) == INVALID
    assert g(P, 1024, 4, 2, 1, 512, NULL, P, NULL, P + 4, NULL, NULL) == INVALID


def test_merge_argument_checks(lib):
    f = lib.dsa_merge_topk_stable
    assert f(P, 0, 1024, 512, P, NULL, NULL, NULL) == OK
    assert f(NULL, 4, 1024, 512, P, NULL, NULL, NULL) == INVALID
    assert f(P, 4, 1024, 512, NULL, NULL, NULL, NULL) == INVALID
    assert f(P, 4, 256, 512, P, NULL, NULL, NULL) == INVALID      # C < K
    assert f(P, 4, 1026, 512, P, NULL, NULL, NULL) == INVALID     # C % 4
    assert f(P, 4, 1024, 500, P, NULL, NULL, NULL) == UNSUPPORTED


def test_convert_argument_checks(lib):
    f = lib.dsa_convert_index_compact
    base = dict(ids=P, rows=4, K=512, S=2, I=1, bt=P, reqs=4, mb=8, bs=64, r2q=NULL, slots=P)

    def call(**kw):
        a = {**base, **kw}
        return f(a["ids"], a["rows"], a["K"], a["S"], a["I"], a["bt"], a["reqs"], a["mb"],
                 a["bs"], a["r2q"], a["slots"], NULL, NULL, NULL)
    assert call(rows=0) == OK
    assert call(ids=NULL) == INVALID
    assert call(bt=NULL) == INVALID
    assert call(slots=NULL) == INVALID
    assert call(bs=0) == INVALID
    assert call(reqs=0) == INVALID
    assert call(mb=0) == INVALID
    assert call(S=0) == UNSUPPORTED
    assert call(I=0) == UNSUPPORTED
    assert call(K=64) == UNSUPPORTED


def test_fused_argument_checks(lib):
    f = lib.dsa_indexer_fused

    def call(logits=P, ld=1024, rows=4, S=4, I=1, K=512, ends=P, bt=P, reqs=4, mb=8, bs=64,
             ids=P, slots=P, cand=NULL):
        return f(logits, ld, rows, S, I, K, NULL, ends, bt, reqs, mb, bs, NULL, ids, NULL, slots,
                 NULL, NULL, cand, NULL, NULL)
    assert call(rows=0, logits=NULL, ends=NULL, bt=NULL, ids=NULL, slots=NULL) == OK
    assert call(logits=NULL) == INVALID
    assert call(ends=NULL) == INVALID
    assert call(bt=NULL) == INVALID
    assert call(ids=NULL) == INVALID
    assert call(slots=NULL) == INVALID
    assert call(cand=P + 8) == INVALID
    assert call(ld=1023) == INVALID
    assert call(bs=0) == INVALID
    assert call(S=9) == UNSUPPORTED        # above the portable cluster size
    assert call(S=0) == UNSUPPORTED
    assert call(K=4096) == UNSUPPORTED


def test_zero_rows_accepts_null_arrays(lib):
    assert lib.dsa_shard_topk(NULL, 64, 0, 2, 1, 512, NULL, NULL, NULL, NULL, NULL) == OK
    assert lib.dsa_merge_topk_stable(NULL, 0, 1024, 512, NULL, NULL, NULL, NULL) == OK
    assert lib.dsa_lse_combine(NULL, NULL, 2, 0, 4, 64, NULL, NULL, NULL, NULL) == OK


def test_combine_argument_checks(lib):
    f = lib.dsa_lse_combine
    assert f(P, P, 4, 0, 8, 64, P, NULL, NULL, NULL) == OK
    assert f(NULL, P, 4, 2, 8, 64, P, NULL, NULL, NULL) == INVALID
    assert f(P, NULL, 4, 2, 8, 64, P, NULL, NULL, NULL) == INVALID
    assert f(P, P, 4, 2, 8, 64, NULL, NULL, NULL, NULL) == INVALID
    assert f(P, P, 4, 2, 8, 60, P, NULL, NULL, NULL) == INVALID        # D % 8
    assert f(P, P, 4, 2, 0, 64, P, NULL, NULL, NULL) == INVALID
    assert f(P + 2, P, 4, 2, 8, 64, P, NULL, NULL, NULL) == INVALID
    assert f(P, P, 0, 2, 8, 64, P, NULL, NULL, NULL) == UNSUPPORTED
    assert f(P, P, 65, 2, 8, 64, P, NULL, NULL, NULL) == UNSUPPORTED


def test_slot_mapping_argument_checks(lib):
    f = lib.dsa_slot_mapping
    assert f(NULL, NULL, 0, 4, 1, NULL, 2, 8, 64, NULL, NULL, NULL) == OK      # n == 0
    assert f(NULL, NULL, 5, 4, 1, P, 2, 8, 64, P, NULL, NULL) == INVALID
    assert f(P, NULL, 5, 4, 1, NULL, 2, 8, 64, P, NULL, NULL) == INVALID
    assert f(P, NULL, 5, 4, 1, P, 2, 8, 64, NULL, NULL, NULL) == INVALID
    assert f(P, NULL, -1, 4, 1, P, 2, 8, 64, P, NULL, NULL) == INVALID
    assert f(P, NULL, 5, 4, 1, P, 0, 8, 64, P, NULL, NULL) == INVALID          # reqs
    assert f(P, NULL, 5, 4, 1, P, 2, 0, 64, P, NULL, NULL) == INVALID          # max_blocks
    assert f(P, NULL, 5, 4, 1, P, 2, 8, 0, P, NULL, NULL) == INVALID           # block size
    assert f(P, NULL, 5, 0, 1, P, 2, 8, 64, P, NULL, NULL) == UNSUPPORTED
    assert f(P, NULL, 5, 65, 1, P, 2, 8, 64, P, NULL, NULL) == UNSUPPORTED
    assert f(P, NULL, 5, 4, 0, P, 2, 8, 64, P, NULL, NULL) == UNSUPPORTED
    assert f(P, NULL, 5, 64, 2 ** 30, P, 2, 8, 64, P, NULL, NULL) == UNSUPPORTED  # I*S


def test_sparse_mla_decode_argument_checks(lib):
    f = lib.dsa_sparse_mla_decode
    ok = (P, P, 1000, P, P, 2, 4, 128, 2048, 0.07, P, P, NULL, NULL)
    assert f(*ok[:5], 0, *ok[6:]) == OK                                   # rows == 0
    for i, bad in [(0, NULL), (1, NULL), (3, NULL), (4, NULL), (10, NULL), (11, NULL),
                   (0, P + 8), (1, P + 4), (10, P + 2), (2, 0), (8, 0),
                   (9, float("inf")), (9, float("nan")), (5, -1)]:
        args = list(ok)
        args[i] = bad
        assert f(*args) == INVALID, (i, bad)
    for i, bad in [(6, 0), (6, 65), (7, 96), (7, 32), (7, 16)]:
        args = list(ok)
        args[i] = bad
        assert f(*args) == UNSUPPORTED, (i, bad)


def test_binding_rejects_cpu_tensors():
    import torch
    import dsa_sparse_indexer_gb300 as dsa
    x = torch.zeros(2, 4, 16)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.shard_topk(x, torch.zeros(4, dtype=torch.int32), 512, 1)
    with pytest.raises(ValueError, match="CUDA"):
        dsa.lse_combine(torch.zeros(2, 1, 1, 8, dtype=torch.bfloat16),
                        torch.zeros(2, 1, 1))


def test_product_code_does_not_import_the_oracle():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "dsa_sparse_indexer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
