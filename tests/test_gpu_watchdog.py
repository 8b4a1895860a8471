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
    ensure_built()
    q, k, v = qkv_inputs.normal_qkv(1, 2, 512, 512, 128, seed=13, dtype=torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    try:
        assert pkg.attn_test_set_hook(1, 20_000_000) == pkg.ATTN_OK  # 20 ms limit
        pkg.attention(qd, kd, vd, causal=True, out_dtype=torch.float32)
        assert pkg.attn_check_status(None) == pkg.ATTN_ERR_TIMEOUT
        # the status word was cleared by the read
        assert pkg.attn_check_status(None) == pkg.ATTN_OK
    finally:
        assert pkg.attn_test_set_hook(0, DEFAULT_TIMEOUT_NS) == pkg.ATTN_OK
    o, lse = pkg.attention(qd, kd, vd, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    assert_bf16_parity(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref)
