"""Tensors of more than 2^31 elements: every path must form its offsets in 64
bits.

K and V hold 5 heads x N = 2^22 + 17 keys x 128 (2.68e9 elements each, 5.4 GB
in bf16), so every key of head 4 lies past element 2^31.  K is zero except
one key j_h = N - 1 - 5h per head, whose first component is 12; q is the
unit vector e_0 and the scale is 1, so that key scores exactly 12 and every
other key 0.  (The key sits in the last tile of its head: keys that follow
the jump of the maximum add increments about 2^-17 times the accumulator,
whose fp32 rounding would otherwise build up over thousands of keys.)  V is
0.5 everywhere except row j_h, which holds w_c = (c + 1) / 64.  Every value
is exact in bf16, and the answer has a closed form (fp64):

    o_c = ((N - 1) 0.5 + e^12 w_c) / (N - 1 + e^12),   lse = ln(N - 1 + e^12)

A wrong (wrapped) offset would read a zero key or the wrong value row and
miss it by far more than the tolerance.  Each path is checked: the
tensor-core kernel (one query row per head), split-KV and the fp32 kernel."""
import math

import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu

H, N, D = 5, (1 << 22) + 17, 128
S_STAR = 12.0


def _inputs(dtype):
    q = torch.zeros((1, H, 1, D), dtype=dtype, device="cuda")
    q[..., 0] = 1.0
    k = torch.zeros((1, H, N, D), dtype=dtype, device="cuda")
    v = torch.full((1, H, N, D), 0.5, dtype=dtype, device="cuda")
    w = (torch.arange(D, dtype=torch.float64) + 1) / 64
    for h in range(H):
        j = N - 1 - 5 * h
        k[0, h, j, 0] = S_STAR
        v[0, h, j, :] = w.to(dtype).cuda()
    assert (H - 1) * N * D > 2 ** 31  # the last head lies past element 2^31
    return q, k, v, w.numpy()


def _expected(w):
    e = math.exp(S_STAR)
    o = ((N - 1) * 0.5 + e * w) / (N - 1 + e)
    return o, math.log(N - 1 + e)


def _check(o, lse, w, tol):
    o_ref, lse_ref = _expected(w)
    o = o.double().cpu().numpy().reshape(H, D)
    assert np.abs(o - o_ref[None, :]).max() <= tol
    assert np.abs(lse.double().cpu().numpy().reshape(H) - lse_ref).max() <= 1e-4 * lse_ref


@pytest.mark.parametrize("path", ["tensor_core", "splitkv"])
def test_bf16_beyond_2_31_elements(path):
    ensure_built()
    q, k, v, w = _inputs(torch.bfloat16)
    if path == "tensor_core":
        o, lse = pkg.attention(q, k, v, scale=1.0, out_dtype=torch.float32)
    else:
        o, lse = pkg.attention_splitkv(q, k, v, scale=1.0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    _check(o, lse, w, 2e-3)
    del q, k, v
    torch.cuda.empty_cache()


def test_fp32_beyond_2_31_elements():
    ensure_built()
    q, k, v, w = _inputs(torch.float32)
    o, lse = pkg.attention(q, k, v, scale=1.0)
    torch.cuda.synchronize()
    _check(o, lse, w, 1e-5)
    del q, k, v
    torch.cuda.empty_cache()
