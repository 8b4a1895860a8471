"""attn_fwd_splitkv_noalloc: the split-KV forward for callers that cannot
allocate device memory -- code running inside an allocator or a memory-pool
callback, or a serving path that forbids allocation.  Instead of a
caller-provided workspace it uses a scratch array that is part of the
library's device image.

Each call is checked against attn_fwd_splitkv with a caller workspace, on
the same inputs and split count, within the tolerances of the other parity
tests.  Two calls are made in a row with different problems, so the second
one also shows that what the first left in the shared scratch does not leak
into its result.  This file runs last in the suite and also passes on its own
in a fresh process."""
import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import ensure_built


def _noalloc(q, k, v, causal, code, n_splits, out_dtype):
    B, H, Sq, d = q.shape
    Skv = k.shape[2]
    o = torch.empty((B, H, Sq, d), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    st = pkg.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code,
                                      n_splits, None)
    assert st == pkg.ATTN_OK, pkg.attn_strerror(st)
    return o, lse


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_on_two_calls():
    ensure_built()
    cases = [
        # B, H, Sq, Skv, d, causal, dtype, out dtype, code, max abs, mean abs
        (2, 8, 3, 5000, 128, False, torch.bfloat16, torch.float32, pkg.ATTN_BF16_OUT_F32,
         1e-2, 1e-3),
        (1, 4, 8, 1024, 32, True, torch.float32, torch.float32, pkg.ATTN_F32, 1e-5, 1e-5),
    ]
    for seed, (B, H, Sq, Skv, d, causal, dt, odt, code, tol_max, tol_mean) in enumerate(cases):
        q, k, v = (t.to(dt).cuda() for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=30 + seed))
        st, n_splits, _ = pkg.attn_splitkv_plan(B, H, Sq, Skv, d, code)
        assert st == pkg.ATTN_OK
        o, lse = _noalloc(q, k, v, causal, code, n_splits, odt)
        o_ws, lse_ws = pkg.attention_splitkv(q, k, v, causal=causal, out_dtype=odt,
                                             n_splits=n_splits)
        torch.cuda.synchronize()
        assert pkg.attn_check_status(None) == pkg.ATTN_OK
        err = (o.double() - o_ws.double()).abs()
        assert err.max().item() <= tol_max and err.mean().item() <= tol_mean
        lerr = (lse.double() - lse_ws.double()).abs() / lse_ws.double().abs().clamp(min=1.0)
        assert lerr.max().item() <= 1e-5
        # and both agree with the oracle on one head
        o_ref, lse_ref = oracle.attention(q[0, 0].cpu(), k[0, 0].cpu(), v[0, 0].cpu(),
                                          causal=causal)
        assert np.abs(o[0, 0].double().cpu().numpy() - o_ref).max() <= tol_max


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Checked on the host before any launch, so the fake (never touched)
    addresses are safe on any machine."""
    ensure_built()
    B, H, Sq, d, n = 64, 64, 8, 128, 4  # 4 * 4 * 4096 * 8 * 129 bytes > 8 MiB
    st, need = pkg.attn_splitkv_workspace_size(B, H, Sq, d, n)
    assert st == pkg.ATTN_OK and need > pkg.NOALLOC_SCRATCH_BYTES
    gib4 = 1 << 32  # addresses 4 GiB apart, so that no two arguments overlap
    st = pkg.attn_fwd_splitkv_noalloc(1 * gib4, 2 * gib4, 3 * gib4, 4 * gib4, 5 * gib4, B, H,
                                      Sq, 64, d, 0, 0.0, pkg.ATTN_BF16, n, None)
    assert st == pkg.ATTN_ERR_SCRATCH_LIMIT
    assert "scratch" in pkg.attn_strerror(st)


def test_noalloc_size_errors_on_the_host():
    """Host-side checks before any launch (fake, never touched addresses, far
    enough apart that no two arguments overlap): a problem with no keys needs
    no scratch, so its size never meets the scratch limit; a problem whose
    scratch size does not fit in 64 bits is an invalid argument, as it is
    for attn_fwd_splitkv."""
    ensure_built()
    gib4 = 1 << 32
    B, H, Sq, d, n = 64, 64, 8, 128, 4  # more than the scratch holds, had it keys
    if torch.cuda.is_available():
        # with a device the call goes on to write o = 0, lse = -inf: real buffers
        o = torch.full((B, H, Sq, d), 7.0, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros((B, H, Sq), dtype=torch.float32, device="cuda")
        q = torch.zeros_like(o)
        st = pkg.attn_fwd_splitkv_noalloc(q.data_ptr(), None, None, o.data_ptr(),
                                          lse.data_ptr(), B, H, Sq, 0, d, 0, 0.0,
                                          pkg.ATTN_BF16, n, None)
        torch.cuda.synchronize()
        assert st == pkg.ATTN_OK
        assert bool((o == 0).all()) and bool(torch.isneginf(lse).all())
    else:
        # without one the device check refuses it, after the size checks
        st = pkg.attn_fwd_splitkv_noalloc(1 * gib4, 2 * gib4, 3 * gib4, 4 * gib4, 5 * gib4,
                                          B, H, Sq, 0, d, 0, 0.0, pkg.ATTN_BF16, n, None)
        assert st == pkg.ATTN_ERR_UNSUPPORTED_DEVICE
    big = 1 << 60
    B = H = 46340  # B * H just below 2^31; 256 splits of 524280 rows overflow
    st = pkg.attn_fwd_splitkv_noalloc(1 * big, 2 * big, 3 * big, 4 * big, 5 * big, B, H,
                                      524280, 64, 128, 0, 0.0, pkg.ATTN_BF16, 256, None)
    assert st == pkg.ATTN_ERR_INVALID_ARG
    st = pkg.attn_fwd_splitkv(1 * big, 2 * big, 3 * big, 4 * big, 5 * big, B, H, 524280, 64,
                              128, 0, 0.0, pkg.ATTN_BF16, 256, 6 * big, 1 << 40, None)
    assert st == pkg.ATTN_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_later_calls_leave_free_memory_unchanged():
    """Once a call of the same kind has run on the device (which loads the
    library's device code there, the scratch array included), further calls
    take nothing from the device's free memory, and give the same bits."""
    ensure_built()
    B, H, Sq, Skv, d = 2, 8, 3, 5000, 128
    q, k, v = (t.to(torch.bfloat16).cuda()
               for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=40))
    st, n_splits, _ = pkg.attn_splitkv_plan(B, H, Sq, Skv, d, pkg.ATTN_BF16)
    assert st == pkg.ATTN_OK
    outs = [(torch.empty((B, H, Sq, d), dtype=torch.bfloat16, device="cuda"),
             torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")) for _ in range(3)]

    def call(o, lse):
        st = pkg.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          o.data_ptr(), lse.data_ptr(), B, H, Sq, Skv, d, 0,
                                          0.0, pkg.ATTN_BF16, n_splits, None)
        assert st == pkg.ATTN_OK, pkg.attn_strerror(st)

    call(*outs[0])  # set-up call
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    call(*outs[1])
    call(*outs[2])
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
