"""Host-only checks of the C ABI: the library loads without a GPU, exports
every function include/attn.h declares, and rejects invalid arguments before
any CUDA call (attn_validate never dereferences its pointers)."""
import math
import os
import re

import pytest

import online_softmax_forward_gb300 as pkg
from online_softmax_forward_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return pkg.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


def defined_symbols(path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_every_declared_function_is_exported(lib):
    declared = header_functions()
    assert len(declared) >= 8
    assert sorted(pkg.exported_symbols()) == declared
    syms = defined_symbols(pkg.library_path())
    for name in declared:
        assert name in syms, name
        assert hasattr(lib, name)


def test_abi_version_and_messages(lib):
    assert pkg.attn_abi_version() == 1
    for s in range(6):
        assert pkg.attn_strerror(s)
    assert "unknown" in pkg.attn_strerror(99)


# fake, never-dereferenced, 16-byte aligned addresses
Q, K, V, O, L = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000


def val(q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, Sq=64, Skv=64, d=64, causal=0,
        scale=0.0, dtype=pkg.ATTN_BF16):
    return pkg.attn_validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype)


def test_valid_arguments_pass(lib):
    assert val() == pkg.ATTN_OK
    assert val(dtype=pkg.ATTN_F32, d=16) == pkg.ATTN_OK
    assert val(dtype=pkg.ATTN_F32, d=128) == pkg.ATTN_OK
    assert val(dtype=pkg.ATTN_F16, d=128, causal=1) == pkg.ATTN_OK
    assert val(lse=None) == pkg.ATTN_OK
    assert val(scale=0.125) == pkg.ATTN_OK


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(o=None),
    dict(q=Q + 8), dict(o=O + 2), dict(lse=L + 2),
    dict(d=48), dict(d=32), dict(dtype=pkg.ATTN_F32, d=24), dict(dtype=7), dict(dtype=-1),
    dict(B=-1), dict(Sq=-5), dict(Skv=-1), dict(d=0), dict(causal=2),
    dict(scale=float("nan")), dict(scale=float("inf")),
    dict(o=Q),                      # output aliases an input
    dict(lse=K + 64),               # lse inside k
    dict(lse=O + 16),               # lse inside o
], ids=lambda kw: ",".join("%s=%s" % i for i in kw.items()))
def test_invalid_arguments_rejected(lib, kw):
    assert val(**kw) == pkg.ATTN_ERR_INVALID_ARG


def test_empty_problems_are_valid(lib):
    # nothing to read or write: pointers may be NULL
    assert val(q=None, k=None, v=None, o=None, lse=None, B=0) == pkg.ATTN_OK
    assert val(q=None, k=None, v=None, o=None, lse=None, Sq=0) == pkg.ATTN_OK
    # no keys: o and lse are still written, k/v may be NULL
    assert val(k=None, v=None, Skv=0) == pkg.ATTN_OK


def test_blocked_entry_rejects_bad_tiles(lib):
    f = pkg.load_library().attn_fwd_f32_blocked
    for bq, bkv in ((0, 16), (16, 0), (129, 16), (16, 257), (128, 256)):
        assert f(Q, K, V, O, L, 1, 1, 64, 64, 128, 0, 0.0, bq, bkv, None) == \
            pkg.ATTN_ERR_INVALID_ARG


def test_hook_rejects_unknown_values(lib):
    assert pkg.attn_test_set_hook(5, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_test_set_hook(0, 0) == pkg.ATTN_OK


def test_default_scale():
    assert pkg.default_scale(128) == 1.0 / math.sqrt(128)
