"""Out-of-bounds writes, checked without a sanitizer: every output buffer of
each path is placed inside a larger allocation whose head and tail are
filled with NaN (16-byte aligned guard bands), the call runs on ragged
shapes (rows past a tile, keys past a tile, rows with no visible key), and
the guard bands must come back untouched while the output in between
matches the oracle."""
import math

import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import (assert_bf16_parity, assert_f32_parity, assert_rounded_output,
                      ensure_built)

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side


def guarded(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((GUARD + n + GUARD,), math.nan, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


def check_guards(buf, n):
    head, tail = buf[:GUARD], buf[GUARD + n:]
    assert torch.isnan(head).all().item() and torch.isnan(tail).all().item(), "guard band written"


@pytest.mark.parametrize("case", [
    # B, H, Sq, Skv, d, causal, in dtype, out dtype
    (1, 3, 300, 517, 128, True, torch.bfloat16, torch.bfloat16),
    (2, 1, 517, 300, 128, True, torch.bfloat16, torch.float32),   # rows with no visible key
    (1, 2, 333, 129, 64, False, torch.float16, torch.float16),
    (1, 2, 77, 200, 32, True, torch.float32, torch.float32),      # CUDA-core path
])
def test_attn_fwd_writes_only_its_outputs(case):
    ensure_built()
    B, H, Sq, Skv, d, causal, idt, odt = case
    q, k, v = (t.to(idt).cuda() for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Sq + Skv))
    obuf, o = guarded((B, H, Sq, d), odt)
    lbuf, lse = guarded((B, H, Sq), torch.float32)
    pkg.attention(q, k, v, causal=causal, out_dtype=odt, out=o, lse=lse)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    check_guards(obuf, o.numel())
    check_guards(lbuf, lse.numel())
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal)
    on, ln = o.double().cpu().numpy(), lse.double().cpu().numpy()
    if idt == torch.float32:
        assert_f32_parity(on, ln, o_ref, lse_ref)
    elif odt == torch.float32:
        assert_bf16_parity(on, ln, o_ref, lse_ref)
    else:
        assert_rounded_output(on, o_ref, odt)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(ln), fin)


@pytest.mark.parametrize("case", [
    (1, 2, 1, 1000, 128, False, torch.bfloat16),
    (2, 1, 9, 333, 64, True, torch.float32),
])
def test_splitkv_writes_only_its_outputs_and_workspace(case):
    ensure_built()
    B, H, Sq, Skv, d, causal, idt = case
    q, k, v = (t.to(idt).cuda() for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Skv))
    code = pkg.ATTN_F32 if idt == torch.float32 else pkg.ATTN_BF16_OUT_F32
    n_splits = 5
    st, need = pkg.attn_splitkv_workspace_size(B, H, Sq, d, n_splits)
    assert st == pkg.ATTN_OK
    wbuf, ws = guarded((need // 4,), torch.float32)
    obuf, o = guarded((B, H, Sq, d), torch.float32)
    lbuf, lse = guarded((B, H, Sq), torch.float32)
    st = pkg.attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code, n_splits,
                              ws.data_ptr(), need, None)
    assert st == pkg.ATTN_OK
    torch.cuda.synchronize()
    check_guards(wbuf, ws.numel())
    check_guards(obuf, o.numel())
    check_guards(lbuf, lse.numel())
    o_ref, _ = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal)
    tol = 1e-5 if idt == torch.float32 else 1e-2
    assert np.abs(o.double().cpu().numpy() - o_ref).max() <= tol
