"""attn_shutdown: the library gives up its per-device state and sets it up
again on the next call.  The library's streams and events of the host-staged
path are destroyed; the cached capability check, SM count, kernel
shared-memory limits, status-word and scratch addresses are forgotten.
Calls made after a shutdown (two in a row, which is harmless) must give
results bit-identical to the same calls made before it: tensor-core,
fp32, split-KV, no-alloc and host-staged (chunked, so its streams are
really re-created)."""
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import qkv_inputs
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


def _staged(q, k, v, causal, code):
    B, H, S, d = q.shape
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty((B, H, S, d), dtype=q.dtype).pin_memory()
    lh = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    do_ = torch.empty((B, H, S, d), dtype=q.dtype, device="cuda")
    dl = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    st = pkg.attn_fwd_staged(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                             lh.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                             do_.data_ptr(), dl.data_ptr(), B, H, S, S, d, int(causal), 0.0,
                             code, torch.cuda.current_stream().cuda_stream)
    assert st == pkg.ATTN_OK
    torch.cuda.synchronize()
    return oh.clone(), lh.clone()


def _noalloc(q, k, v):
    B, H, Sq, d = q.shape
    o = torch.empty((B, H, Sq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    st = pkg.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, Sq, k.shape[2], d, 0, 0.0,
                                      pkg.ATTN_BF16_OUT_F32, 3, None)
    assert st == pkg.ATTN_OK
    return o, lse


def _all_paths():
    bf = [t.to(torch.bfloat16) for t in qkv_inputs.normal_qkv(2, 8, 1024, 1024, 128, seed=21)]
    f32 = [t.cuda() for t in qkv_inputs.normal_qkv(1, 3, 200, 300, 64, seed=22)]
    dec = [t.to(torch.bfloat16).cuda() for t in qkv_inputs.normal_qkv(2, 4, 1, 3000, 128, seed=23)]
    out = {
        "tc": pkg.attention(*(t.cuda() for t in bf), causal=True),
        "f32": pkg.attention(*f32, causal=True),
        "splitkv": pkg.attention_splitkv(*dec),
        "noalloc": _noalloc(*dec),
    }
    out["staged"] = _staged(*bf, True, pkg.ATTN_BF16)  # 8 MiB of input: chunked
    torch.cuda.synchronize()
    return out


def test_calls_after_shutdown_match_calls_before():
    ensure_built()
    before = _all_paths()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    assert pkg.attn_shutdown() == pkg.ATTN_OK
    assert pkg.attn_shutdown() == pkg.ATTN_OK
    after = _all_paths()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    for name in before:
        (o0, l0), (o1, l1) = before[name], after[name]
        assert torch.equal(o0, o1) and torch.equal(l0, l1), name
    # the staged result is the device call's
    assert torch.equal(after["staged"][0], after["tc"][0].cpu())
