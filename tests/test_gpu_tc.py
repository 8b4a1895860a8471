"""bf16/fp16 tensor-core path against the fp64 oracle run on the same
16-bit-rounded inputs.  Tolerances (fp32 output): max abs <= 1e-2, mean abs
<= 1e-3, lse within 1e-4 * max(1, |lse|); 16-bit output: within 1e-2 plus one
unit in the last place of the rounded oracle value."""
import math

import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import (assert_bf16_parity, assert_lse_close, assert_rounded_output, cast_like,
                      ensure_built, run)

pytestmark = pytest.mark.gpu

SMALL = [
    # B, H, Sq, Skv, d, causal
    (1, 1, 128, 128, 128, True),
    (1, 2, 256, 256, 128, True),
    (1, 2, 384, 384, 128, False),
    (2, 2, 1000, 1000, 128, True),   # ragged: 1000 = 7*128 + 104
    (1, 3, 300, 517, 128, True),     # Sq < Skv, bottom-right causal
    (1, 3, 517, 300, 128, True),     # Sq > Skv: leading rows see no key
    (1, 2, 517, 300, 128, False),
    (1, 1, 1, 1, 128, False),
    (1, 1, 5, 700, 128, False),      # decode-like
    (1, 2, 640, 640, 64, True),      # d = 64
    (2, 1, 333, 129, 64, False),
    (4, 40, 300, 300, 128, True),    # 320 units: three snake rounds over the SMs
    (2, 80, 260, 260, 64, False),    # 320 units at d = 64, ragged tail tiles
]


def _id(c):
    return "B%dH%d_%dx%d_d%d_%s" % (c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", SMALL, ids=_id)
def test_small_shapes_fp32_out(case, dtype):
    B, H, Sq, Skv, d, causal = case
    q, k, v = qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Sq + Skv + d, dtype=dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o, lse = run(q, k, v, causal, dtype=dtype, out_dtype=torch.float32)
    assert_bf16_parity(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", SMALL[:6], ids=_id)
def test_small_shapes_16bit_out(case, dtype):
    B, H, Sq, Skv, d, causal = case
    q, k, v = qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Sq * 3 + Skv, dtype=dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o, lse = run(q, k, v, causal, dtype=dtype)
    assert_rounded_output(o, o_ref, dtype)
    assert_lse_close(lse, lse_ref, 1e-4)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_large_scores_stay_finite(dtype):
    """The large-score exercise (scores x 50, q multiplied by 50): rows are
    dominated by one or two keys, so the 16-bit rounding of the dominant
    probability would show in full if the normaliser did not sum exactly the
    rounded probabilities that multiply V.  The standard bounds hold: max abs
    <= 1e-2, mean abs <= 1e-3, lse within 1e-4 * max(1, |lse|)."""
    q, k, v = qkv_inputs.normal_qkv(1, 2, 256, 512, 128, seed=9)
    q = (q * 50).to(dtype)
    k, v = k.to(dtype), v.to(dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False)
    o, lse = run(q, k, v, False, dtype=dtype, out_dtype=torch.float32)
    assert np.all(np.isfinite(o))
    assert_bf16_parity(o, lse, o_ref, lse_ref)


def test_rising_maximum_forces_rescale():
    """Scores that grow along the keys (q = 1, key sums ramping to 60) make
    each row's running maximum rise by more than the lazy-rescale threshold
    on every key tile, so the accumulator rescale runs on each of them."""
    B, H, S, d = 1, 2, 1024, 128
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(21)
    q = torch.ones(B, H, S, d)
    ramp = torch.linspace(0.0, 60.0, S) / (scale * d)
    k = ramp[None, None, :, None].expand(B, H, S, d) + 0.05 * torch.randn(B, H, S, d, generator=g)
    v = torch.randn(B, H, S, d, generator=g)
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
        o, lse = run(q, k, v, causal, dtype=torch.bfloat16, out_dtype=torch.float32)
        assert_bf16_parity(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_masked_keys_never_set_the_row_max(d, dtype):
    """The softmax takes a tile's row maximum from the TMEM load itself, which
    covers all 128 keys of the tile; on a diagonal or tail tile some of them
    are masked and must not count.  Two inputs make any masked key that did
    count push the running maximum so far above the visible scores that
    their probabilities flush to zero:
    * causal, 256 keys, keys 192-255 scoring ~300 above the rest: rows 128-191
      see the first 64 keys of the diagonal tile only, next to masked keys
      300 higher;
    * non-causal, 200 keys all scoring about -300: the 56 key slots past the
      end of the tail tile load as zeros, i.e. score 0, 300 above every
      visible key.
    Both must match the oracle at the standard bounds."""
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(33)
    cases = []
    q = torch.ones(1, 2, 256, d)
    k = 0.05 * torch.randn(1, 2, 256, d, generator=g)
    k[:, :, 192:] += 300.0 / (scale * d)
    cases.append((q, k, torch.randn(1, 2, 256, d, generator=g), True))
    q = torch.ones(1, 2, 130, d)
    k = -300.0 / (scale * d) + 0.05 * torch.randn(1, 2, 200, d, generator=g)
    cases.append((q, k, torch.randn(1, 2, 200, d, generator=g), False))
    for q, k, v, causal in cases:
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
        o, lse = run(q, k, v, causal, dtype=dtype, out_dtype=torch.float32)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        assert_bf16_parity(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("skv", [8192, 8193])
@pytest.mark.parametrize("out32", [False, True])
def test_output_store_paths_at_the_key_threshold(skv, out32):
    """With up to 8192 keys (d = 128) the unit epilogue writes O through shared
    memory, two rows or half rows per store instruction; with more keys it
    stores each row directly.  Both paths, with 16-bit and fp32 output, on
    ragged query rows (300 = 2 x 128 + 44) and 4 heads."""
    q, k, v = qkv_inputs.normal_qkv(1, 4, 300, skv, 128, seed=skv + 3 * out32)
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
        if out32:
            o, lse = run(q, k, v, causal, dtype=torch.bfloat16, out_dtype=torch.float32)
            assert_bf16_parity(o, lse, o_ref, lse_ref)
        else:
            o, lse = run(q, k, v, causal, dtype=torch.bfloat16, out_dtype=torch.bfloat16)
            assert_rounded_output(o, o_ref, torch.bfloat16)
            assert_lse_close(lse, lse_ref, 1e-4)


def _sampled_parity(B, H, S, d, seed, n_random, heads=None, rows_per_head=None, causal=True,
                    dtype=torch.bfloat16):
    ensure_built()
    q, k, v = qkv_inputs.normal_qkv(B, H, S, S, d, seed=seed, dtype=dtype)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o32, lse = pkg.attention(qd, kd, vd, causal=causal, out_dtype=torch.float32)
    o16, lse16 = pkg.attention(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    # properties of every row
    assert torch.isfinite(o32).all() and torch.isfinite(lse).all()
    if causal:
        # row 0 sees key 0 only: its output is v[0] (exactly, once rounded to bf16)
        assert torch.allclose(o32[:, :, 0], vd[:, :, 0].float(), rtol=1e-6, atol=0)
        assert torch.equal(o16[:, :, 0], vd[:, :, 0])
    assert torch.equal(lse, lse16)
    vmin = vd.float().amin(dim=2, keepdim=True)
    vmax = vd.float().amax(dim=2, keepdim=True)
    assert bool(((o32 >= vmin - 1e-3) & (o32 <= vmax + 1e-3)).all())  # convex combination
    # sampled rows against the oracle
    BH = B * H
    heads = range(BH) if heads is None else heads
    qh, kh, vh = (t.reshape(BH, S, d) for t in (q, k, v))
    rows, o_parts, l_parts = [], [], []
    for bh in heads:
        rs = qkv_inputs.sample_rows(S, n_random, seed=1000 + bh)
        o_b, l_b = oracle.attention_rows(qh[bh:bh + 1], kh[bh:bh + 1], vh[bh:bh + 1],
                                         [(0, i) for i in rs], causal=causal)
        rows += [(bh, i) for i in rs]
        o_parts.append(o_b)
        l_parts.append(l_b)
    o_ref, lse_ref = np.concatenate(o_parts), np.concatenate(l_parts)
    o32h = o32.reshape(BH, S, d).double().cpu().numpy()
    o16h = o16.reshape(BH, S, d).double().cpu().numpy()
    lseh = lse.reshape(BH, S).double().cpu().numpy()
    idx = np.asarray(rows)
    got = o32h[idx[:, 0], idx[:, 1]]
    got_l = lseh[idx[:, 0], idx[:, 1]]
    mx, mean = assert_bf16_parity(got, got_l, o_ref, lse_ref)
    assert_rounded_output(o16h[idx[:, 0], idx[:, 1]], o_ref, dtype)
    return mx, mean, len(rows)


def test_b1_h32_s8192_d128_causal_sampled():
    """B=1, H=32, Sq=Skv=8192, d=128, bf16, causal, scale 1/sqrt(128):
    every row checked for the properties above; ~200 stratified rows per
    head (all tile boundaries) against the oracle."""
    mx, mean, n = _sampled_parity(1, 32, 8192, 128, seed=0, n_random=64)
    print("c4 sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_b1_h32_s8192_d128_fp16_causal_sampled():
    """The same workload in fp16 (fp16 P for P.V, the other instruction
    descriptor): every row checked for the properties; stratified rows of
    eight heads against the oracle."""
    mx, mean, n = _sampled_parity(1, 32, 8192, 128, seed=3, n_random=32,
                                  heads=(0, 5, 10, 15, 16, 21, 26, 31), dtype=torch.float16)
    print("fp16 8k sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_b1_h64_s8192_d64_causal_sampled():
    """d = 64 at full size (P in tensor memory, six-stage ring; 64 heads, so
    head groups of 8): every row checked for the properties; stratified rows
    of eight heads against the oracle."""
    mx, mean, n = _sampled_parity(1, 64, 8192, 64, seed=4, n_random=32,
                                  heads=(0, 7, 8, 23, 40, 47, 56, 63))
    print("d=64 8k sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_b1_h64_s32768_d128_causal_sampled():
    """B=1, H=64, Sq=Skv=32768, d=128, bf16, causal: every row checked for
    the properties; ~520 stratified rows in each of four heads against the
    oracle."""
    mx, mean, n = _sampled_parity(1, 64, 32768, 128, seed=0, n_random=8,
                                  heads=(0, 21, 42, 63))
    print("c5 sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_grouped_schedule_noncausal_sampled():
    """B=1, H=20, Sq=Skv=32768, d=128, non-causal: the K and V of all heads
    (336 MB) exceed the L2, so the units are scheduled in head groups of 3
    (the last group holds 2); sampled rows of heads in the first, a middle
    and the last group against the oracle."""
    mx, mean, n = _sampled_parity(1, 20, 32768, 128, seed=2, n_random=4, heads=(0, 10, 19),
                                  causal=False)
    print("grouped non-causal sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_unequal_head_groups_sampled():
    """B=1, H=7, Sq=Skv=32768, d=128, non-causal: 7 heads have no divisor
    covering a round of units and their K and V (112 MB) exceed what L2
    holds, so the schedule takes groups of 2 heads with a last group of 1;
    sampled rows of a head in the first, a middle and the last group."""
    mx, mean, n = _sampled_parity(1, 7, 32768, 128, seed=6, n_random=4, heads=(0, 3, 6),
                                  causal=False)
    print("unequal groups sampled rows %d: max %.3e mean %.3e" % (n, mx, mean))


def test_deterministic():
    q, k, v = (t.cuda() for t in qkv_inputs.normal_qkv(1, 4, 1000, 1000, 128, 5,
                                                        dtype=torch.bfloat16))
    ensure_built()
    o1, l1 = pkg.attention(q, k, v, causal=True)
    o2, l2 = pkg.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_staged_host_buffers_match_device_call():
    """attn_fwd_staged (host buffers, copies inside the call) equals attn_fwd."""
    ensure_built()
    B, H, S, d = 1, 2, 640, 128
    q, k, v = qkv_inputs.normal_qkv(B, H, S, S, d, seed=4, dtype=torch.bfloat16)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty((B, H, S, d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    do_ = torch.empty((B, H, S, d), dtype=torch.bfloat16, device="cuda")
    dl = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    st = pkg.attn_fwd_staged(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                             lh.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                             do_.data_ptr(), dl.data_ptr(), B, H, S, S, d, 1, 0.0,
                             pkg.ATTN_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == pkg.ATTN_OK
    torch.cuda.synchronize()
    o_dev, l_dev = pkg.attention(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_dev.cpu()) and torch.equal(lh, l_dev.cpu())


@pytest.mark.parametrize("case", [
    # B, H, Sq, Skv, d, causal, dtype: >= 4 MiB of input, so the call runs in chunks
    (2, 8, 1024, 1024, 128, True, torch.bfloat16),
    (1, 5, 700, 1300, 64, True, torch.float16),
    (2, 3, 600, 600, 64, False, torch.float32),
])
def test_staged_chunked_matches_device_call(case):
    """Large host-staged calls are cut into up to four chunks of (batch, head)
    slices of unequal sizes (16 slices: 3, 5, 6, 2; 5: 1, 2, 1, 1; 6: 1, 2,
    2, 1) on two library streams; the result is the same as the device call,
    and work queued on the caller's stream afterwards sees it complete."""
    ensure_built()
    B, H, Sq, Skv, d, causal, dt = case
    q, k, v = (t.to(dt) for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Sq + H))
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty((B, H, Sq, d), dtype=dt).pin_memory()
    lh = torch.empty((B, H, Sq), dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    do_ = torch.empty((B, H, Sq, d), dtype=dt, device="cuda")
    dl = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    code = pkg.dtype_code(dt)
    st = pkg.attn_fwd_staged(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(),
                             lh.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                             do_.data_ptr(), dl.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0,
                             code, s.cuda_stream)
    assert st == pkg.ATTN_OK
    with torch.cuda.stream(s):
        after = do_.float().sum()  # queued on the caller's stream after the call
    s.synchronize()
    assert pkg.attn_check_status(s.cuda_stream) == pkg.ATTN_OK
    o_dev, l_dev = pkg.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(oh, o_dev.cpu()) and torch.equal(lh, l_dev.cpu())
    assert torch.equal(do_, o_dev)
    assert after.item() == o_dev.float().sum().item()
