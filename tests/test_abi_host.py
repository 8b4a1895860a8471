"""Host-only checks of the C ABI: the library loads without a GPU, exports
every function include/attn.h declares (and the test library also those of
include/attn_test.h), and rejects invalid arguments before any CUDA call
(attn_validate never dereferences its pointers)."""
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


def header_functions(name="attn.h"):
    text = open(os.path.join(ROOT, "include", name)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:ATTN_API\s+)?(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(",
                                 text, flags=re.M)))


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


def test_product_library_exports_nothing_else(lib):
    """libattn.so exports the functions of attn.h and no other function of
    its own: the test-only entry points are absent, and nothing internal
    (C++ symbols of the attn namespace, kernels) is visible."""
    syms = defined_symbols(pkg.library_path())
    for name in header_functions("attn_test.h"):
        assert name not in syms, name
    ours = {s for s in syms if s.startswith("attn") or "4attn" in s}
    assert ours == set(header_functions())


def test_test_library_exports_both_headers(lib):
    test_only = header_functions("attn_test.h")
    assert sorted(pkg.test_exported_symbols()) == test_only
    assert set(test_only) == {"attn_fwd_f32_blocked", "attn_test_set_hook"}
    syms = defined_symbols(pkg.test_library_path())
    for name in header_functions() + test_only:
        assert name in syms, name
    tl = pkg.load_test_library()
    for name in test_only:
        assert hasattr(tl, name)


def test_abi_version_and_messages(lib):
    assert pkg.attn_abi_version() == 1
    for s in range(8):
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
    f = pkg.load_test_library().attn_fwd_f32_blocked
    for bq, bkv in ((0, 16), (16, 0), (129, 16), (16, 257), (128, 256)):
        assert f(Q, K, V, O, L, 1, 1, 64, 64, 128, 0, 0.0, bq, bkv, None) == \
            pkg.ATTN_ERR_INVALID_ARG


def test_hook_rejects_unknown_values(lib):
    assert pkg.attn_test_set_hook(5, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_test_set_hook(0, 0) == pkg.ATTN_OK


def test_default_scale():
    assert pkg.default_scale(128) == 1.0 / math.sqrt(128)


# ------------------------------------------------------------------ split-KV and merge
def test_splitkv_workspace_size(lib):
    st, n = pkg.attn_splitkv_workspace_size(2, 4, 8, 32, 3)
    assert st == pkg.ATTN_OK and n == 4 * 3 * 2 * 4 * 8 * 33
    st, n = pkg.attn_splitkv_workspace_size(0, 4, 8, 32, 3)
    assert st == pkg.ATTN_OK and n == 0
    for args in ((2, 4, 8, 48, 3), (2, 4, 8, 32, 0), (2, 4, 8, 32, 257), (-1, 4, 8, 32, 1)):
        assert pkg.attn_splitkv_workspace_size(*args)[0] == pkg.ATTN_ERR_INVALID_ARG


W = 0x100000  # fake workspace address, far from the other fake pointers


def skv(q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, Sq=8, Skv=64, d=32, causal=0, scale=0.0,
        dtype=pkg.ATTN_F32, n_splits=2, ws=W, ws_bytes=1 << 20):
    return pkg.attn_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype,
                                n_splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw", [
    dict(n_splits=0), dict(n_splits=257), dict(ws=None), dict(ws=W + 8),
    dict(ws_bytes=4 * 2 * 2 * 8 * 33 - 4),   # one float short
    dict(ws=Q), dict(ws=O - 64),               # workspace overlaps q / o
    dict(d=48), dict(dtype=9), dict(causal=3), dict(q=Q + 4), dict(Sq=524281),
], ids=lambda kw: ",".join("%s=%s" % i for i in kw.items()))
def test_splitkv_rejects_invalid_arguments(lib, kw):
    assert skv(**kw) == pkg.ATTN_ERR_INVALID_ARG


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return True


def test_splitkv_accepts_every_width_and_empty_problems(lib):
    # Valid arguments pass validation and then stop at the device check.  The
    # fake addresses must never reach a kernel, so this part runs only on a
    # host without a GPU.
    if not _no_gpu():
        pytest.skip("valid calls with fake pointers would launch on this host")
    for dt in (pkg.ATTN_F32, pkg.ATTN_BF16, pkg.ATTN_F16):
        for d in (16, 32, 64, 128):
            assert skv(d=d, dtype=dt) == pkg.ATTN_ERR_UNSUPPORTED_DEVICE
    assert skv(B=0, q=None, k=None, v=None, o=None, lse=None, ws=None) == pkg.ATTN_OK
    assert skv(Sq=0, ws=None) == pkg.ATTN_OK


def merge_call(po=0x200000, pl=0x300000, n=3, rows=16, d=32, o=0x400000, lse=0x500000,
               out=pkg.ATTN_F32):
    return pkg.attn_merge(po, pl, n, rows, d, o, lse, out, None)


@pytest.mark.parametrize("kw", [
    dict(n=0), dict(n=4097), dict(rows=-1), dict(rows=1 << 31), dict(d=0), dict(out=pkg.ATTN_BF16_OUT_F32), dict(out=7),
    dict(po=None), dict(pl=None), dict(o=None), dict(po=0x200002), dict(o=0x400001),
    dict(o=0x200000 + 64),          # output inside the partial outputs
    dict(lse=0x300000),             # lse on top of the partial lse
], ids=lambda kw: ",".join("%s=%s" % i for i in kw.items()))
def test_merge_rejects_invalid_arguments(lib, kw):
    assert merge_call(**kw) == pkg.ATTN_ERR_INVALID_ARG


def test_merge_empty_rows_is_noop(lib):
    assert merge_call(rows=0, po=None, pl=None, o=None, lse=None) == pkg.ATTN_OK


def test_shutdown_without_a_device_reports_cuda_error(lib):
    """On a host without a GPU there is no current device to release."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host has a GPU: covered by the GPU tests")
    assert pkg.attn_shutdown() == pkg.ATTN_ERR_CUDA


def test_torch_wrappers_reject_host_tensors_before_any_call(lib):
    """The wrappers hand raw pointers to the kernels: CPU tensors are refused
    on the host, before anything is launched."""
    import torch
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pkg.attention(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        pkg.attention_splitkv(q, q, q, n_splits=1)
    with pytest.raises(ValueError, match="CUDA"):
        pkg.merge(torch.zeros(2, 4, 64), torch.zeros(2, 4))


def test_checked_library_exports_the_test_library_functions(lib):
    """libattn_checked.so, the bounds-checking build, carries the same entry
    points as the test library."""
    syms = defined_symbols(pkg.checked_library_path())
    for name in header_functions() + header_functions("attn_test.h"):
        assert name in syms, name
    cl = pkg.load_checked_library()
    assert cl.attn_abi_version() == 1
    assert cl.attn_strerror(pkg.ATTN_ERR_BOUNDS).decode().startswith("bounds-checking build")
