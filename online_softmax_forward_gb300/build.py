"""Build libattn.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in parallel to an object under _build/, then two
shared libraries are linked next to this file:

* libattn.so -- the product: exports the functions of include/attn.h only
  (hidden visibility for everything else);
* libattn_test.so -- the same objects, with attn_api.cu compiled a second
  time with ATTN_TEST_EXPORTS, so that it also exports the test-only entry
  points of include/attn_test.h;
* libattn_checked.so -- the bounds-checking build: every source compiled
  with ATTN_BOUNDS_CHECK (and the test exports), so that the kernels test
  each global index and TMA coordinate before using it and report a failed
  test through the status word instead of touching memory out of bounds.

The CUDA runtime is linked statically (nvcc's default), so the libraries
need only the driver at run time; the tensor-map encoder is fetched from the
driver at first use.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libattn.so")
TEST_LIB = os.path.join(HERE, "libattn_test.so")
CHECKED_LIB = os.path.join(HERE, "libattn_checked.so")
SOURCES = ["attn_api.cu", "attn_f32.cu", "attn_splitkv.cu", "attn_tc.cu"]
# (source, object name, extra flags) of the test library's own objects
TEST_SOURCES = [("attn_api.cu", "attn_api_test.o", ["-DATTN_TEST_EXPORTS"])]
# ... and of the bounds-checking library's, one per source
CHECKED_SOURCES = [(src, src.replace(".cu", "_checked.o"),
                    ["-DATTN_BOUNDS_CHECK"] + (["-DATTN_TEST_EXPORTS"] if src == "attn_api.cu"
                                               else []))
                   for src in SOURCES]
HEADERS = ["attn_internal.h", "sm100_ptx.cuh"]
PUBLIC_HEADERS = ["attn.h", "attn_test.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return (ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-Xcompiler", "-fvisibility=hidden",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
            + list(extra))


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = ([src] + [os.path.join(INCLUDE, h) for h in PUBLIC_HEADERS]
            + [os.path.join(CSRC, h) for h in HEADERS])
    return any(os.path.getmtime(d) > t for d in deps)


def _link(lib: str, objs) -> None:
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + list(objs)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        print(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Builds the three libraries (only what is stale); returns the product's path."""
    os.makedirs(BUILD, exist_ok=True)
    objs, jobs = {}, []
    units = ([(src, src.replace(".cu", ".o"), []) for src in SOURCES] + TEST_SOURCES
             + CHECKED_SOURCES)
    for src, oname, fl in units:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, oname)
        objs[oname] = o
        if force or _stale(o, s):
            jobs.append([nvcc()] + _flags(list(extra_flags) + fl) + ["-c", s, "-o", o])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for %s" % cmd[-3])
    product = [objs[src.replace(".cu", ".o")] for src in SOURCES]
    test_set = product[:]
    for src, oname, _ in TEST_SOURCES:  # the test build replaces the product object
        test_set[SOURCES.index(src)] = objs[oname]
    if jobs or not os.path.exists(LIB) or force:
        _link(LIB, product)
    if jobs or not os.path.exists(TEST_LIB) or force:
        _link(TEST_LIB, test_set)
    if jobs or not os.path.exists(CHECKED_LIB) or force:
        _link(CHECKED_LIB, [objs[t[1]] for t in CHECKED_SOURCES])
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
