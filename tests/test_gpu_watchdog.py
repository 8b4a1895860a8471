"""Failure detection of the tensor-core kernel without a GPU fault.

Every mbarrier wait of the kernel is bounded.  attn_test_set_hook(1, ns)
makes the next launches skip one internal completion signal (the first
score-tile commit of CTA 0), so one wait can never be satisfied: it gives up
after `ns`, the CTA stops its roles, drains its own copies and MMAs, frees
tensor memory and returns, and attn_check_status reports ATTN_ERR_TIMEOUT.
The context stays usable: the next call without the hook is exact again."""
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import assert_bf16_parity, ensure_built

pytestmark = pytest.mark.gpu

DEFAULT_TIMEOUT_NS = 1_000_000_000


def test_expired_wait_reports_timeout_and_context_recovers():
    """Runs on the test library (libattn_test.so), the only one that exports
    the hook; attn_fwd and attn_check_status are that library's too, since
    the hook and the status word are per library."""
    ensure_built()
    tl = pkg.load_test_library()
    B, H, S, d = 1, 2, 512, 128
    q, k, v = qkv_inputs.normal_qkv(B, H, S, S, d, seed=13, dtype=torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty((B, H, S, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")

    def fwd():
        st = tl.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                         lse.data_ptr(), B, H, S, S, d, 1, 0.0, pkg.ATTN_BF16_OUT_F32, None)
        assert st == pkg.ATTN_OK

    try:
        assert tl.attn_test_set_hook(1, 20_000_000) == pkg.ATTN_OK  # 20 ms limit
        fwd()
        assert tl.attn_check_status(None) == pkg.ATTN_ERR_TIMEOUT
        # the status word was cleared by the read
        assert tl.attn_check_status(None) == pkg.ATTN_OK
    finally:
        assert tl.attn_test_set_hook(0, DEFAULT_TIMEOUT_NS) == pkg.ATTN_OK
    fwd()
    torch.cuda.synchronize()
    assert tl.attn_check_status(None) == pkg.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    assert_bf16_parity(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref)
