"""Python binding of libattn.so -- exact attention forward with online softmax
for GB300 (sm_103a).

The functions named like the C ABI (``attn_fwd``, ``attn_validate``, ...)
take raw pointers and sizes and only marshal arguments; ``attention`` is the
convenience call on PyTorch CUDA tensors (it allocates the outputs with torch
and calls ``attn_fwd``).  Every step of the computation runs in the library's
CUDA kernels; if the library is missing this module raises instead of
computing anything another way.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED_DEVICE", "ATTN_ERR_LAUNCH",
    "ATTN_ERR_TIMEOUT", "ATTN_ERR_CUDA", "ATTN_ERR_SCRATCH_LIMIT", "ATTN_ERR_BOUNDS",
    "NOALLOC_SCRATCH_BYTES",
    "ATTN_F32", "ATTN_BF16", "ATTN_F16", "ATTN_BF16_OUT_F32", "ATTN_F16_OUT_F32",
    "AttnError", "library_path", "load_library", "exported_symbols",
    "test_library_path", "load_test_library", "test_exported_symbols",
    "checked_library_path", "load_checked_library",
    "attn_fwd", "attn_validate", "attn_fwd_f32_blocked", "attn_fwd_staged",
    "attn_check_status", "attn_strerror", "attn_abi_version", "attn_test_set_hook",
    "attn_splitkv_workspace_size", "attn_splitkv_plan", "attn_fwd_splitkv", "attn_merge",
    "attn_fwd_splitkv_noalloc", "attn_shutdown",
    "attention", "attention_f32_blocked", "attention_splitkv", "merge", "dtype_code",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED_DEVICE = 2
ATTN_ERR_LAUNCH = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_CUDA = 5
ATTN_ERR_SCRATCH_LIMIT = 6
ATTN_ERR_BOUNDS = 7  # the bounds-checking build (libattn_checked.so) only
NOALLOC_SCRATCH_BYTES = 8 << 20  # the fixed scratch of attn_fwd_splitkv_noalloc

ATTN_F32 = 0
ATTN_BF16 = 1
ATTN_F16 = 2
ATTN_BF16_OUT_F32 = 3
ATTN_F16_OUT_F32 = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None
_test_lib = None
_checked_lib = None

# (name, restype, argtypes) of every symbol declared in include/attn.h
# (libattn.so) and, in _TEST_SIGS, in include/attn_test.h (libattn_test.so only)
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SIGS = [
    ("attn_fwd", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    ("attn_validate", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I]),
    ("attn_fwd_staged", _I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                             _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    ("attn_check_status", _I, [_P]),
    ("attn_strerror", ctypes.c_char_p, [_I]),
    ("attn_abi_version", _I, []),
    ("attn_splitkv_workspace_size", _I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    ("attn_splitkv_plan", _I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I),
                               ctypes.POINTER(ctypes.c_size_t)]),
    ("attn_fwd_splitkv", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P,
                              ctypes.c_size_t, _P]),
    ("attn_merge", _I, [_P, _P, _I, ctypes.c_int64, _I, _P, _P, _I, _P]),
    ("attn_fwd_splitkv_noalloc", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                                      _P]),
    ("attn_shutdown", _I, []),
]
_TEST_SIGS = [
    ("attn_fwd_f32_blocked", _I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    ("attn_test_set_hook", _I, [_I, ctypes.c_uint64]),
]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, _strerror_safe(status), status))


def library_path() -> str:
    return os.environ.get("ATTN_GB300_LIB", os.path.join(_HERE, "libattn.so"))


def test_library_path() -> str:
    return os.environ.get("ATTN_GB300_TEST_LIB", os.path.join(_HERE, "libattn_test.so"))


def _open(path, sigs, what):
    if not os.path.exists(path):
        raise ImportError("%s not found at %s: build it with "
                          "online_softmax_forward_gb300.build.build()" % (what, path))
    lib = ctypes.CDLL(path)
    for name, res, args in sigs:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_library():
    """Load libattn.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    if _lib is None:
        _lib = _open(library_path(), _SIGS, "libattn.so")
    return _lib


def load_test_library():
    """Load libattn_test.so: the product's functions plus the test-only entry
    points of include/attn_test.h.  It is a separate library with its own
    state (status word, hook): call the functions of a test on it alone."""
    global _test_lib
    if _test_lib is None:
        _test_lib = _open(test_library_path(), _SIGS + _TEST_SIGS, "libattn_test.so")
    return _test_lib


def checked_library_path() -> str:
    return os.path.join(_HERE, "libattn_checked.so")


def load_checked_library():
    """Load libattn_checked.so: the test library built with ATTN_BOUNDS_CHECK,
    whose kernels test every global index and TMA coordinate before using it
    (attn_check_status then reports ATTN_ERR_BOUNDS).  A separate library
    with its own state, like the test library."""
    global _checked_lib
    if _checked_lib is None:
        _checked_lib = _open(checked_library_path(), _SIGS + _TEST_SIGS, "libattn_checked.so")
    return _checked_lib


def exported_symbols():
    return [s[0] for s in _SIGS]


def test_exported_symbols():
    return [s[0] for s in _TEST_SIGS]


def _strerror_safe(status: int) -> str:
    try:
        return load_library().attn_strerror(int(status)).decode()
    except Exception:  # pragma: no cover
        return "status %d" % status


def _check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)
    return status


# ------------------------------------------------------------------ raw ABI
def attn_fwd(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, stream):
    return load_library().attn_fwd(q, k, v, o, lse, B, H, Sq, Skv, d, int(causal),
                                   float(scale), dtype, stream)


def attn_validate(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype):
    return load_library().attn_validate(q, k, v, o, lse, B, H, Sq, Skv, d, int(causal),
                                        float(scale), dtype)


def attn_fwd_f32_blocked(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, block_q,
                         block_kv, stream):
    """Test library only (include/attn_test.h)."""
    return load_test_library().attn_fwd_f32_blocked(q, k, v, o, lse, B, H, Sq, Skv, d,
                                                    int(causal), float(scale), block_q,
                                                    block_kv, stream)


def attn_fwd_staged(q_host, k_host, v_host, o_host, lse_host, dq, dk, dv, do_, dlse,
                    B, H, Sq, Skv, d, causal, scale, dtype, stream):
    return load_library().attn_fwd_staged(q_host, k_host, v_host, o_host, lse_host, dq, dk,
                                           dv, do_, dlse, B, H, Sq, Skv, d, int(causal),
                                           float(scale), dtype, stream)


def attn_check_status(stream):
    return load_library().attn_check_status(stream)


def attn_strerror(status):
    return load_library().attn_strerror(int(status)).decode()


def attn_abi_version():
    return load_library().attn_abi_version()


def attn_shutdown():
    return load_library().attn_shutdown()


def attn_test_set_hook(hook, timeout_ns=0):
    """Test library only (include/attn_test.h): arms the hook of
    libattn_test.so, which affects that library's attn_fwd alone."""
    return load_test_library().attn_test_set_hook(int(hook), int(timeout_ns))


def attn_splitkv_workspace_size(B, H, Sq, d, n_splits):
    """Returns (status, bytes)."""
    n = ctypes.c_size_t(0)
    st = load_library().attn_splitkv_workspace_size(B, H, Sq, d, n_splits, ctypes.byref(n))
    return st, n.value


def attn_splitkv_plan(B, H, Sq, Skv, d, dtype):
    """Returns (status, n_splits, workspace_bytes)."""
    n = ctypes.c_int(0)
    b = ctypes.c_size_t(0)
    st = load_library().attn_splitkv_plan(B, H, Sq, Skv, d, dtype, ctypes.byref(n),
                                          ctypes.byref(b))
    return st, n.value, b.value


def attn_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, n_splits,
                     workspace, workspace_bytes, stream):
    return load_library().attn_fwd_splitkv(q, k, v, o, lse, B, H, Sq, Skv, d, int(causal),
                                           float(scale), dtype, int(n_splits), workspace,
                                           int(workspace_bytes), stream)


def attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Skv, d, causal, scale, dtype, n_splits,
                             stream):
    """attn_fwd_splitkv with the library's fixed device scratch instead of a
    workspace: for callers that cannot allocate (see include/attn.h)."""
    return load_library().attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Sq, Skv, d,
                                                   int(causal), float(scale), dtype,
                                                   int(n_splits), stream)


def attn_merge(o_parts, lse_parts, n_parts, rows, d, o, lse, out_dtype, stream):
    return load_library().attn_merge(o_parts, lse_parts, int(n_parts), int(rows), int(d), o,
                                     lse, int(out_dtype), stream)


# ------------------------------------------------------------------ torch helpers
def dtype_code(in_dtype, out_dtype=None) -> int:
    """attn_dtype for torch input/output dtypes."""
    import torch
    if in_dtype == torch.float32:
        if out_dtype not in (None, torch.float32):
            raise ValueError("fp32 inputs give fp32 output")
        return ATTN_F32
    if in_dtype == torch.bfloat16:
        if out_dtype in (None, torch.bfloat16):
            return ATTN_BF16
        if out_dtype == torch.float32:
            return ATTN_BF16_OUT_F32
    if in_dtype == torch.float16:
        if out_dtype in (None, torch.float16):
            return ATTN_F16
        if out_dtype == torch.float32:
            return ATTN_F16_OUT_F32
    raise ValueError("unsupported dtypes %s -> %s" % (in_dtype, out_dtype))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, S, d]")
    B, H, Sq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("shape mismatch q %s k %s v %s" % (tuple(q.shape), tuple(k.shape),
                                                            tuple(v.shape)))
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    _device_of(q, k, v)
    return B, H, Sq, k.shape[2], d


def _device_of(*tensors):
    """The one CUDA device all tensors live on; raises otherwise (the kernels
    are handed raw device pointers)."""
    dev = None
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors (got %s)" % t.device)
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors on different devices: %s and %s" % (dev, t.device))
    return dev


def _check_out(t, shape, dtype, dev, name):
    """A caller-provided output must match exactly what the call writes."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s tensor of shape %s" % (name, dtype, tuple(shape)))
    if not t.is_cuda or t.device != dev:
        raise ValueError("%s must be on %s" % (name, dev))


def attention(q, k, v, causal: bool = False, scale: float | None = None, out_dtype=None,
              return_lse: bool = True, out=None, lse=None, stream=None):
    """O (and LSE) for contiguous CUDA tensors q [B,H,Sq,d], k/v [B,H,Skv,d].

    ``out_dtype`` = torch.float32 with bf16/fp16 inputs selects the fp32-output
    variant.  Outputs are allocated with torch unless ``out`` / ``lse`` are
    given."""
    import torch
    B, H, Sq, Skv, d = _shapes(q, k, v)
    code = dtype_code(q.dtype, out_dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share a dtype")
    odt = {ATTN_F32: torch.float32, ATTN_BF16: torch.bfloat16, ATTN_F16: torch.float16,
           ATTN_BF16_OUT_F32: torch.float32, ATTN_F16_OUT_F32: torch.float32}[code]
    if out is None:
        out = torch.empty((B, H, Sq, d), dtype=odt, device=q.device)
    _check_out(out, (B, H, Sq, d), odt, q.device, "out")
    if return_lse and lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_out(lse, (B, H, Sq), torch.float32, q.device, "lse")
    sc = 0.0 if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                      lse.data_ptr() if lse is not None else None, B, H, Sq, Skv, d, causal,
                      sc, code, _stream_handle(stream))
    _check(st, "attn_fwd")
    return (out, lse) if return_lse else out


def attention_f32_blocked(q, k, v, block_q: int, block_kv: int, causal: bool = False,
                          scale: float | None = None, stream=None):
    """fp32 path with explicit tile sizes (block-size invariance tests;
    runs in the test library, include/attn_test.h)."""
    import torch
    B, H, Sq, Skv, d = _shapes(q, k, v)
    out = torch.empty((B, H, Sq, d), dtype=torch.float32, device=q.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = attn_fwd_f32_blocked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, Sq, Skv, d, causal, sc, block_q,
                                  block_kv, _stream_handle(stream))
    _check(st, "attn_fwd_f32_blocked")
    return out, lse


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def attention_splitkv(q, k, v, causal: bool = False, scale: float | None = None,
                      out_dtype=None, n_splits: int | None = None, workspace=None,
                      stream=None):
    """Split-KV forward (few query rows, long key sequences).  The workspace is
    a torch uint8 CUDA tensor, allocated here unless given; ``n_splits`` is
    the library's choice unless given.  Returns (o, lse)."""
    import torch
    B, H, Sq, Skv, d = _shapes(q, k, v)
    code = dtype_code(q.dtype, out_dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share a dtype")
    if n_splits is None:
        with torch.cuda.device(q.device):
            st, n_splits, _ = attn_splitkv_plan(B, H, Sq, Skv, d, code)
        _check(st, "attn_splitkv_plan")
    st, need = attn_splitkv_workspace_size(B, H, Sq, d, n_splits)
    _check(st, "attn_splitkv_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if not workspace.is_contiguous() or _device_of(workspace) != q.device:
        raise ValueError("workspace must be a contiguous tensor on %s" % q.device)
    odt = {ATTN_F32: torch.float32, ATTN_BF16: torch.bfloat16, ATTN_F16: torch.float16,
           ATTN_BF16_OUT_F32: torch.float32, ATTN_F16_OUT_F32: torch.float32}[code]
    out = torch.empty((B, H, Sq, d), dtype=odt, device=q.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    with torch.cuda.device(q.device):
        st = attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, H, Sq, Skv, d, causal, sc, code, n_splits,
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(stream))
    _check(st, "attn_fwd_splitkv")
    return out, lse


def merge(o_parts, lse_parts, out_dtype=None, stream=None):
    """attn_merge on torch tensors: o_parts [n, rows, d] fp32, lse_parts
    [n, rows] fp32 -> (o [rows, d], lse [rows])."""
    import torch
    if o_parts.dim() != 3 or lse_parts.shape != o_parts.shape[:2]:
        raise ValueError("o_parts [n, rows, d] and lse_parts [n, rows] expected")
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("partial results are fp32")
    o_parts, lse_parts = o_parts.contiguous(), lse_parts.contiguous()
    _device_of(o_parts, lse_parts)
    n, rows, d = o_parts.shape
    odt = torch.float32 if out_dtype is None else out_dtype
    code = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16, torch.float16: ATTN_F16}[odt]
    out = torch.empty((rows, d), dtype=odt, device=o_parts.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        st = attn_merge(o_parts.data_ptr(), lse_parts.data_ptr(), n, rows, d, out.data_ptr(),
                        lse.data_ptr(), code, _stream_handle(stream))
    _check(st, "attn_merge")
    return out, lse
