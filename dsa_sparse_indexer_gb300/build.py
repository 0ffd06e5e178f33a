"""Build libdsa.so (the C-ABI library) in-tree for sm_103a.

Each .cu file under csrc/ is compiled in parallel to an object file, then the
objects are linked into `_build/libdsa.so` next to this file.  Nothing is
installed; the Python binding loads the library from that path.

    python -m dsa_sparse_indexer_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found; the CUDA library cannot be built")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    files.append(os.path.join(INCLUDE, "dsa.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = list(extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


STALLED_COPY_TEST_LIB = os.path.join(BUILD, "libdsa_stalled_copy_test.so")


def build_stalled_copy_test(force: bool = False) -> str:
    """A test-only library, separate from libdsa.so: the local top-K, the
    sparse MLA decode and the indexer logits entry points (shard_topk.cu,
    attention.cu, indexer_logits.cu) built with DSA_TEST_STALLED_COPY, where
    the top-K's staging wait and the logits' first MMA also wait on an
    mbarrier that no copy completes and the attention's stage barriers expect
    one arrival that nothing makes, with a short poll bound.  Every real copy
    still lands; the bounded waits run out and the kernels return with
    DSA_FLAG_TIMEOUT set.  Used by the tests of that flag only."""
    srcs = [os.path.join(CSRC, f) for f in ("shard_topk.cu", "attention.cu", "indexer_logits.cu")]
    deps = srcs + [os.path.abspath(__file__), os.path.join(INCLUDE, "dsa.h")] + \
        [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    if (not force and os.path.exists(STALLED_COPY_TEST_LIB) and
            all(os.path.getmtime(f) <= os.path.getmtime(STALLED_COPY_TEST_LIB) for f in deps)):
        return STALLED_COPY_TEST_LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = STALLED_COPY_TEST_LIB + ".tmp"
    cmd = [nvcc(), *ARCH, *FLAGS, "-DDSA_TEST_STALLED_COPY", "-shared", "-cudart", "shared",
           *srcs, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on the stalled-copy test build:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, STALLED_COPY_TEST_LIB)
    return STALLED_COPY_TEST_LIB


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register/smem use")
    a = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if a.ptxas_info else []
    print(build(force=a.force or a.ptxas_info, verbose=a.verbose or a.ptxas_info, extra=extra))
    return 0


if __name__ == "__main__":
    sys.exit(main())
