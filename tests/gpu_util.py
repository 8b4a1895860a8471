"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle element by element."""
from __future__ import annotations

import math

import numpy as np
import torch

import online_softmax_forward_gb300 as pkg
from online_softmax_forward_gb300 import build as lib_build

_built = False


def ensure_built():
    global _built
    if not _built:
        lib_build.build()
        pkg.load_library()
        _built = True


def to_dev(x, dtype):
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x))
    return t.to(dtype).contiguous().cuda()


def run(q, k, v, causal, dtype=torch.float32, out_dtype=None, scale=None, blocks=None):
    """Inputs (numpy or CPU torch) -> CUDA path -> (o, lse) as fp64 numpy.

    The values are first cast to ``dtype`` on the host, so the oracle can be
    run on exactly the values the kernel sees (``cast_like``)."""
    ensure_built()
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    if qd.dim() == 2:
        qd, kd, vd = (t[None, None] for t in (qd, kd, vd))
    if blocks is not None:
        o, lse = pkg.attention_f32_blocked(qd, kd, vd, blocks[0], blocks[1], causal=causal,
                                           scale=scale)
    else:
        o, lse = pkg.attention(qd, kd, vd, causal=causal, scale=scale, out_dtype=out_dtype)
    torch.cuda.synchronize()
    # the blocked entry point runs in the test library, which has its own status word
    lib = pkg.load_test_library() if blocks is not None else pkg.load_library()
    st = lib.attn_check_status(None)
    assert st == pkg.ATTN_OK, pkg.attn_strerror(st)
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def cast_like(x, dtype):
    """The values the kernel receives, widened to fp64."""
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x))
    return t.to(dtype).double().numpy()


def assert_lse_close(lse, lse_ref, rel):
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), finite), "lse finiteness differs"
    assert np.all(lse[~finite] == -math.inf)
    if finite.any():
        err = np.abs(lse[finite] - lse_ref[finite]) / np.maximum(1.0, np.abs(lse_ref[finite]))
        assert err.max() <= rel, "lse rel err %.3e" % err.max()


def assert_f32_parity(o, lse, o_ref, lse_ref, atol=1e-5):
    err = np.abs(o - o_ref)
    assert err.max() <= atol, "max|o err| %.3e > %.1e" % (err.max(), atol)
    assert_lse_close(lse, lse_ref, 1e-5)


def assert_bf16_parity(o, lse, o_ref, lse_ref):
    """bf16/fp16 inputs, fp32 output: max abs <= 1e-2, mean abs <= 1e-3;
    lse within 1e-4 * max(1, |lse|)."""
    err = np.abs(o - o_ref)
    assert err.max() <= 1e-2, "max|o err| %.3e" % err.max()
    assert err.mean() <= 1e-3, "mean|o err| %.3e" % err.mean()
    assert_lse_close(lse, lse_ref, 1e-4)
    return err.max(), err.mean()


def assert_rounded_output(o, o_ref, dtype):
    """16-bit output: within 1e-2 plus one unit in the last place of the
    oracle value rounded to the output type."""
    ref_r = torch.from_numpy(o_ref).to(dtype).double().numpy()
    mant = 7 if dtype == torch.bfloat16 else 10
    mag = np.maximum(np.abs(ref_r), 2.0 ** -14)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - mant)
    err = np.abs(o - o_ref)
    assert np.all(err <= 1e-2 + ulp), "max excess %.3e" % (err - 1e-2 - ulp).max()
    return err.max()
