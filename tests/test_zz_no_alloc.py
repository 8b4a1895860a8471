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
