"""The bounds-checking build (libattn_checked.so: every source compiled with
ATTN_BOUNDS_CHECK) on the shapes that exercise the edges of the index
arithmetic: ragged tails, Sq > Skv and Sq < Skv under the bottom-right
causal mask, d = 64, 16-bit and fp32 outputs, every fp32 launch shape
(one warpgroup with one or two stages, two and four warpgroups splitting
the keys, the d = 64 key-split kernel), runtime tiles of 7 and 13 x 19, split-KV with the warp-per-row
and the CTA-per-row merge, attn_merge and the no-alloc entry point.

Each kernel tests every global-memory index and TMA coordinate it computes
against the extent of its buffer before the access; a failed test sets a bit
of the status word, which attn_check_status reports as ATTN_ERR_BOUNDS.  The
checks stand in for a memory checker, which is not available here: every
call below must come back ATTN_OK, and its result must still match the fp64
oracle within the tolerances of the other parity tests."""
import ctypes

import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import (assert_bf16_parity, assert_f32_parity, assert_lse_close,
                      assert_rounded_output, ensure_built)

pytestmark = pytest.mark.gpu


def _lib():
    ensure_built()
    return pkg.load_checked_library()


def _status(lib):
    st = lib.attn_check_status(None)
    assert st == pkg.ATTN_OK, pkg.attn_strerror(st)


def _inputs(B, H, Sq, Skv, d, dt, seed):
    q, k, v = qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=seed)
    return tuple(t.to(dt) for t in (q, k, v))


def _out(B, H, Sq, d, odt):
    return (torch.empty((B, H, Sq, d), dtype=odt, device="cuda"),
            torch.empty((B, H, Sq), dtype=torch.float32, device="cuda"))


def _np(t):
    return t.double().cpu().numpy()


TC_CASES = [
    # B, H, Sq, Skv, d, causal, input dtype, fp32 output
    (2, 2, 1000, 1000, 128, True, torch.bfloat16, True),   # ragged tail tile
    (1, 3, 517, 300, 128, True, torch.bfloat16, True),     # Sq > Skv: rows with no key
    (1, 3, 300, 517, 128, True, torch.float16, True),      # Sq < Skv
    (1, 2, 640, 640, 64, True, torch.float16, True),       # d = 64
    (2, 1, 333, 129, 64, False, torch.bfloat16, False),    # d = 64, 16-bit output
    (1, 2, 384, 384, 128, False, torch.bfloat16, False),   # 16-bit output
    (4, 40, 300, 300, 128, True, torch.bfloat16, True),    # several schedule rounds
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: "B%dH%d_%dx%d_d%d_%s_%s%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full", str(c[6]).split(".")[-1],
    "_o32" if c[7] else ""))
def test_tensor_core_kernel_checked(case):
    lib = _lib()
    B, H, Sq, Skv, d, causal, dt, out32 = case
    q, k, v = _inputs(B, H, Sq, Skv, d, dt, seed=Sq + 7 * Skv)
    odt = torch.float32 if out32 else dt
    code = pkg.dtype_code(dt, odt)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = _out(B, H, Sq, d, odt)
    st = lib.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, Sq, Skv, d, int(causal), 0.0, code, None)
    assert st == pkg.ATTN_OK
    _status(lib)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    if out32:
        assert_bf16_parity(_np(o), _np(lse), o_ref, lse_ref)
    else:
        assert_rounded_output(_np(o), o_ref, dt)
        assert_lse_close(_np(lse), lse_ref, 1e-4)


F32_CASES = [
    # B, H, Sq, Skv, d, causal: which fp32 launch shape they take
    (1, 1, 64, 64, 32, True),      # one key tile: one warpgroup
    (1, 1, 8, 1024, 32, False),    # few blocks, many key tiles: four warpgroups
    (2, 3, 77, 150, 16, True),     # d = 16: two warpgroups, two stages
    (2, 4, 512, 512, 64, False),   # B=2, H=4, S=512, d = 64: the key-split kernel
    (4, 40, 300, 300, 128, True),  # many blocks: one warpgroup per block
    (1, 3, 70, 40, 64, True),      # Sq > Skv (key-split kernel)
    (1, 2, 33, 2000, 64, True),    # key-split kernel, several tiles per warp, ragged rows
    (4, 40, 300, 300, 64, True),   # d = 64 on a large grid: one warpgroup per block
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "B%dH%d_%dx%d_d%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_fp32_kernel_checked(case):
    lib = _lib()
    B, H, Sq, Skv, d, causal = case
    q, k, v = _inputs(B, H, Sq, Skv, d, torch.float32, seed=Sq + Skv)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = _out(B, H, Sq, d, torch.float32)
    st = lib.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, Sq, Skv, d, int(causal), 0.0, pkg.ATTN_F32, None)
    assert st == pkg.ATTN_OK
    _status(lib)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    assert_f32_parity(_np(o), _np(lse), o_ref, lse_ref)


@pytest.mark.parametrize("blocks", [(7, 7), (13, 19), (1, 1), (128, 64)])
def test_fp32_runtime_tiles_checked(blocks):
    lib = _lib()
    B, H, Sq, Skv, d = 1, 2, 64, 71, 32
    q, k, v = _inputs(B, H, Sq, Skv, d, torch.float32, seed=5)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = _out(B, H, Sq, d, torch.float32)
    st = lib.attn_fwd_f32_blocked(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, Sq, Skv, d, 1, 0.0, blocks[0], blocks[1],
                                  None)
    assert st == pkg.ATTN_OK
    _status(lib)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    assert_f32_parity(_np(o), _np(lse), o_ref, lse_ref)


SPLIT_CASES = [
    # B, H, Sq, Skv, d, causal, dtype, n_splits (> 32: one CTA per row in the merge)
    (2, 8, 3, 5000, 128, False, torch.bfloat16, 7),
    (1, 4, 8, 1024, 32, True, torch.float32, 3),
    (1, 2, 9, 3000, 64, False, torch.float16, 40),
    (1, 1, 1, 33, 16, False, torch.float32, 2),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "B%dH%d_%dx%d_d%d_%s_n%d" % (
    c[0], c[1], c[2], c[3], c[4], str(c[6]).split(".")[-1], c[7]))
def test_splitkv_checked(case):
    lib = _lib()
    B, H, Sq, Skv, d, causal, dt, n = case
    q, k, v = _inputs(B, H, Sq, Skv, d, dt, seed=Skv)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    code = pkg.dtype_code(dt, torch.float32)
    o, lse = _out(B, H, Sq, d, torch.float32)
    need = ctypes.c_size_t(0)
    assert lib.attn_splitkv_workspace_size(B, H, Sq, d, n, ctypes.byref(need)) == pkg.ATTN_OK
    ws = torch.empty(max(need.value, 16), dtype=torch.uint8, device="cuda")
    st = lib.attn_fwd_splitkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code, n,
                              ws.data_ptr(), ws.numel(), None)
    assert st == pkg.ATTN_OK
    _status(lib)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    if dt == torch.float32:
        assert_f32_parity(_np(o), _np(lse), o_ref, lse_ref)
    else:
        assert_bf16_parity(_np(o), _np(lse), o_ref, lse_ref)
    # the no-alloc form of the same call, on the library's fixed scratch
    o2, lse2 = _out(B, H, Sq, d, torch.float32)
    st = lib.attn_fwd_splitkv_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o2.data_ptr(),
                                      lse2.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code,
                                      n, None)
    assert st == pkg.ATTN_OK
    _status(lib)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_merge_checked():
    lib = _lib()
    g = torch.Generator().manual_seed(3)
    n, rows, d = 3, 1000, 96
    po = torch.randn(n, rows, d, generator=g).cuda()
    pl = (torch.randn(n, rows, generator=g) * 4).cuda()
    pl[1, :10] = -float("inf")
    o, lse = torch.empty(rows, d, device="cuda"), torch.empty(rows, device="cuda")
    st = lib.attn_merge(po.data_ptr(), pl.data_ptr(), n, rows, d, o.data_ptr(), lse.data_ptr(),
                        pkg.ATTN_F32, None)
    assert st == pkg.ATTN_OK
    _status(lib)
    o_ref, lse_ref = oracle.merge_partials(po.double().cpu().numpy(), pl.double().cpu().numpy())
    assert np.abs(_np(o) - o_ref).max() <= 1e-5
    assert_lse_close(_np(lse), lse_ref, 1e-5)
