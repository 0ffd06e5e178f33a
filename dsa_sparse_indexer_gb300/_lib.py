"""ctypes loader for libdsa.so, the C-ABI library of the DCP sparse-indexer path.

The library is built in-tree by `dsa_sparse_indexer_gb300.build` (also run by
the repository's top-level build entry point).  There is no fallback: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libdsa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "dsa.h")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA = 0, 1, 2, 3
DSA_FLAG_BOUNDS, DSA_FLAG_TIMEOUT = 1, 2

_p, _i, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64

# Argument types, in the order include/dsa.h declares them.
SIGNATURES = {
    "dsa_status_string": ([_i], ctypes.c_char_p),
    "dsa_version": ([], _i),
    "dsa_shard_topk": ([_p, _i64, _i, _i, _i, _i, _p, _p, _p, _p, _p], _i),
    "dsa_pack_candidates": ([_p, _i64, _p, _i, _i, _i, _i, _p, _p, _p], _i),
    "dsa_shard_topk_pack": ([_p, _i64, _i, _i, _i, _i, _p, _p, _p, _p, _p, _p], _i),
    "dsa_merge_topk_stable": ([_p, _i, _i, _i, _p, _p, _p, _p], _i),
    "dsa_convert_index_compact": ([_p, _i, _i, _i, _i, _p, _i, _i, _i, _p, _p, _p, _p, _p], _i),
    "dsa_indexer_fused": ([_p, _i64, _i, _i, _i, _i, _p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p,
                           _p, _p, _p, _p], _i),
    "dsa_lse_combine": ([_p, _p, _i, _i, _i, _i, _p, _p, _p, _p], _i),
    "dsa_slot_mapping": ([_p, _p, _i, _i, _i, _p, _i, _i, _i, _p, _p, _p], _i),
    "dsa_sparse_mla_decode": ([_p, _p, _i64, _p, _p, _i, _i, _i, _i, ctypes.c_float, _p, _p, _p,
                               _p], _i),
    "dsa_indexer_logits": ([_p, _p, _p, _i64, _p, _i, _i, _i, _p, _p, _p, _i, _i, _i, _p, _i64,
                            _p, _p], _i),
    "dsa_fused_norm_rope": ([_p, _p, _p, _p, ctypes.c_float, _p, _i, _i, _p, _p, _p, _p, _i64,
                             _p, _p], _i),
    "dsa_kv_cache_insert": ([_p, _p, _p, _i, _p, _i64, _p, _p], _i),
    "dsa_indexer_steps_noalloc": ([_p, _i64, _i, _i, _i, _i, _p, _p, _p, _i, _i, _i, _p, _p, _p,
                                   _p, _p, _p], _i),
}

_lib = None


class DSAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the library with argument types set."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libdsa.so not found at {path}; build it with "
            "`python -m dsa_sparse_indexer_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().dsa_status_string(status).decode()


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions include/dsa.h declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(dsa_\w+)\s*\(", text, flags=re.M)


def call(name: str, *args) -> None:
    status = getattr(load(), name)(*args)
    if status != DSA_OK:
        raise DSAError(name, status)
