"""Oracle for exact attention forward -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package.  The product library never does;
nothing here is shared with the CUDA path except the seeded inputs of
``qkv_inputs``.

Contents
--------
``attention`` / ``attention_rows``
    O1: plain fp64 dense attention (C, ``attn_oracle.c``), the definition the
    tiled method reaches up to rounding order -- aiml.sh
    "verify-tiled-attention" ``standard_attention`` and deepnotes
    "flash-attention-implemented-verified-and-measured" ``naive_attention``.
``tiled_attention`` (module ``oracle.tiled``)
    O2: the tiled online-softmax algorithm itself, restated in fp64 NumPy with
    the pages' block sizes and their deliberate "forget to rescale" switch;
    used only to test the algorithm (block-size invariance, the omitted
    rescale, the worked example).
``block_normalised_average`` (module ``oracle.tiled``)
    The knowingly wrong "normalise each block, then average" baseline of
    huhohoo "tiled-online-softmax" ("A failing baseline").
``estimate_hbm_bytes`` (module ``oracle.access``)
    The logical K/V/Q/O access model of aiml.sh "verify-tiled-attention".
``merge_partials`` (module ``oracle.merge``)
    The online-softmax update applied to whole partial results over disjoint
    key sets (huhohoo "tiled-online-softmax", "Online normalization").
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build
from .access import estimate_hbm_bytes  # noqa: F401
from .merge import merge_partials  # noqa: F401
from .tiled import block_normalised_average, tiled_attention  # noqa: F401

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, dbl, ip = ctypes.c_int64, ctypes.c_double, ctypes.c_int
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                        ip, dbl, ip, ip]
        lib.oracle_attn_fwd.restype = ip
        lib.oracle_attn_rows.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                         ip, dbl, ctypes.POINTER(ctypes.c_int64),
                                         i64, ip]
        lib.oracle_attn_rows.restype = ip
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _as_f64(x) -> np.ndarray:
    """Widen any real input (list, numpy array, CPU torch tensor of any float
    dtype) to a contiguous fp64 numpy array without changing its values."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def attention(q, k, v, causal: bool = False, scale: float | None = None,
              subtract_max: bool = True, nthreads: int | None = None):
    """O1 on inputs of shape [..., Sq, d] (q) and [..., Skv, d] (k, v).

    Returns ``(o, lse)`` as fp64 arrays of shapes [..., Sq, d] and [..., Sq].
    ``scale`` defaults to 1/sqrt(d) as on all three pages.  Inputs are widened
    to fp64 first (exact for fp32/bf16/fp16 values)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2] \
            or q.shape[-1] != k.shape[-1]:
        raise ValueError("shape mismatch: q %s k %s v %s" % (q.shape, k.shape, v.shape))
    lead = q.shape[:-2]
    sq, d = q.shape[-2], q.shape[-1]
    skv = k.shape[-2]
    bh = int(np.prod(lead)) if lead else 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = np.zeros(lead + (sq, d), dtype=np.float64)
    lse = np.zeros(lead + (sq,), dtype=np.float64)
    if bh * sq == 0:
        return o, lse
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 bh, sq, skv, d, int(bool(causal)), float(scale),
                                 int(bool(subtract_max)),
                                 nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed (%d)" % rc)
    return o, lse


def attention_rows(q, k, v, rows, causal: bool = False,
                   scale: float | None = None, nthreads: int | None = None):
    """O1 for selected rows only.  q [BH, Sq, d], k/v [BH, Skv, d] (leading
    dims are flattened); ``rows`` is a sequence of (bh, i) pairs.  Returns
    ``(o_rows [n, d], lse_rows [n])`` in the order of ``rows``."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    d = q.shape[-1]
    sq, skv = q.shape[-2], k.shape[-2]
    q = q.reshape(-1, sq, d)
    k = k.reshape(-1, skv, d)
    v = v.reshape(-1, skv, d)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    n = idx.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    if n == 0:
        return o, lse
    rc = _load().oracle_attn_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  q.shape[0], sq, skv, d, int(bool(causal)),
                                  float(scale),
                                  idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                  n, nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attn_rows failed (%d)" % rc)
    return o, lse
