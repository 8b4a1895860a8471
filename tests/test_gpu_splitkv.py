"""Split-KV forward (attn_fwd_splitkv) and the merge of partial results
(attn_merge) on the GPU, through the C ABI, against the fp64 oracle.

Tolerances as for the other paths: fp32 inputs max abs <= 1e-5 and lse
within 1e-5 * max(1, |lse|); 16-bit inputs with fp32 output max abs <= 1e-2,
mean abs <= 1e-3, lse within 1e-4 * max(1, |lse|); 16-bit output within 1e-2
plus one unit in the last place of the rounded oracle value.  The split
count may change only the order of the sums (aiml.sh "verify-tiled-attention"
tile sweep; huhohoo "tiled-online-softmax" block size seven), so every split
count is held to the same bound."""
import math

import numpy as np
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import (assert_bf16_parity, assert_f32_parity, assert_lse_close,
                      assert_rounded_output, cast_like, ensure_built, to_dev)

pytestmark = pytest.mark.gpu


def run_split(q, k, v, causal, dtype=torch.float32, out_dtype=None, n_splits=None, scale=None):
    ensure_built()
    qd, kd, vd = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    if qd.dim() == 2:
        qd, kd, vd = (t[None, None] for t in (qd, kd, vd))
    o, lse = pkg.attention_splitkv(qd, kd, vd, causal=causal, scale=scale, out_dtype=out_dtype,
                                   n_splits=n_splits)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def f32(*xs):
    return [cast_like(x, torch.float32) for x in xs]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("skv", [64, 256, 1024])
@pytest.mark.parametrize("boost", [1.0, 50.0])
@pytest.mark.parametrize("n_splits", [None, 1, 2, 3, 7])
def test_decode_like_fp32(seed, skv, boost, n_splits):
    """Eight query rows, width 32, 64/256/1024 keys, three seeds, no mask
    (huhohoo "tiled-online-softmax" recorded comparison) and q x 50."""
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 8, skv, 32, seed)
    q, k, v = f32(q * boost, k, v)
    o_ref, lse_ref = oracle.attention(q, k, v)
    o, lse = run_split(q, k, v, False, n_splits=n_splits)
    assert_f32_parity(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("case", [
    # B, H, Sq, Skv, d, causal
    (1, 1, 1, 1, 32, False),
    (1, 1, 1, 33, 16, False),
    (2, 3, 1, 1000, 64, True),
    (1, 2, 5, 31, 128, False),
    (1, 2, 9, 700, 32, True),        # two row blocks, ragged
    (2, 1, 17, 300, 64, True),       # three row blocks
    (1, 1, 40, 25, 32, True),        # Sq > Skv: the first 15 rows see no key
    (1, 1, 64, 64, 32, True),        # the single-head causal workload
], ids=lambda c: "B%dH%d_%dx%d_d%d_%s" % (c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
@pytest.mark.parametrize("n_splits", [None, 1, 4, 13])
def test_shapes_fp32(case, n_splits):
    B, H, Sq, Skv, d, causal = case
    q, k, v = f32(*qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Sq + 3 * Skv + d))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o, lse = run_split(q, k, v, causal, n_splits=n_splits)
    assert_f32_parity(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("n_splits", [40, 64, 256])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_more_than_32_splits(n_splits, out_dtype):
    """More than 32 partial results per row: the merge runs one CTA per row
    (up to 32 it runs one warp per row).  5000 keys in splits of a multiple
    of 32 keys give 40, 53 and 157 parts."""
    q, k, v = qkv_inputs.normal_qkv(1, 2, 3, 5000, 64, seed=n_splits, dtype=torch.bfloat16)
    o_ref, lse_ref = oracle.attention(q, k, v)
    o, lse = run_split(q, k, v, False, dtype=torch.bfloat16, out_dtype=out_dtype,
                       n_splits=n_splits)
    if out_dtype == torch.float32:
        assert_bf16_parity(o, lse, o_ref, lse_ref)
    else:
        assert_rounded_output(o, o_ref, torch.bfloat16)
        assert_lse_close(lse, lse_ref, 1e-4)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", [
    (2, 4, 1, 4096, 128, False),
    (1, 4, 8, 1000, 128, True),
    (1, 2, 3, 2048, 64, False),
    (2, 2, 12, 513, 32, True),
], ids=lambda c: "B%dH%d_%dx%d_d%d_%s" % (c[0], c[1], c[2], c[3], c[4], "causal" if c[5] else "full"))
def test_16bit_inputs(case, dtype):
    B, H, Sq, Skv, d, causal = case
    q, k, v = qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Skv + d, dtype=dtype)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o, lse = run_split(q, k, v, causal, dtype=dtype, out_dtype=torch.float32)
    assert_bf16_parity(o, lse, o_ref, lse_ref)
    o16, lse16 = run_split(q, k, v, causal, dtype=dtype)
    assert_rounded_output(o16, o_ref, dtype)
    assert_lse_close(lse16, lse_ref, 1e-4)


def test_long_decode_bf16_sampled_heads():
    """One query row per head against 32768 keys (B=4, H=32, d=128, bf16):
    every output row checked against the oracle on 8 sampled heads."""
    B, H, Skv, d = 4, 32, 32768, 128
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(B, H, n, d, generator=g).to(torch.bfloat16) for n in (1, Skv, Skv))
    o, lse = run_split(q, k, v, False, dtype=torch.bfloat16, out_dtype=torch.float32)
    heads = [(0, 0), (0, 31), (1, 7), (2, 13), (3, 0), (3, 17), (1, 30), (2, 2)]
    for b, h in heads:
        o_ref, lse_ref = oracle.attention(q[b, h], k[b, h], v[b, h])
        assert_bf16_parity(o[b, h], lse[b, h], o_ref, lse_ref)


def test_matches_attn_fwd_and_is_deterministic():
    q, k, v = f32(*qkv_inputs.normal_qkv(2, 2, 6, 2000, 64, seed=4))
    ensure_built()
    qd, kd, vd = (to_dev(x, torch.float32) for x in (q, k, v))
    o1, l1 = pkg.attention_splitkv(qd, kd, vd, causal=True, n_splits=9)
    o2, l2 = pkg.attention_splitkv(qd, kd, vd, causal=True, n_splits=9)
    of, lf = pkg.attention(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1 - of).abs().max().item() <= 1e-5
    assert (l1 - lf).abs().max().item() <= 1e-5


def test_empty_keys_and_empty_batch():
    ensure_built()
    q = torch.randn(1, 2, 3, 32, device="cuda")
    k = torch.empty(1, 2, 0, 32, device="cuda")
    o, lse = pkg.attention_splitkv(q, k, k, n_splits=2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and torch.all(lse == -math.inf).item()
    z = torch.empty(0, 2, 3, 32, device="cuda")
    o, lse = pkg.attention_splitkv(z, torch.empty(0, 2, 5, 32, device="cuda"),
                                   torch.empty(0, 2, 5, 32, device="cuda"), n_splits=2)
    assert o.numel() == 0


def test_plan_fills_the_device():
    ensure_built()
    st, n, ws = pkg.attn_splitkv_plan(1, 32, 1, 32768, 128, pkg.ATTN_BF16)
    assert st == pkg.ATTN_OK and 1 <= n <= 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 32 * n >= sms  # every SM gets at least one partial block
    st2, ws2 = pkg.attn_splitkv_workspace_size(1, 32, 1, 128, n)
    assert st2 == pkg.ATTN_OK and ws2 == ws


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("bounds", [[(0, 100), (100, 101), (101, 777)],
                                    [(500, 777), (0, 500)], [(0, 777)],
                                    # 41 parts: the one-CTA-per-row merge
                                    [(19 * i, 19 * i + 19) for i in range(40)] + [(760, 777)]])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_of_key_shards(bounds, out_dtype):
    """Partial results over key shards (computed by attn_fwd on each shard)
    merged on the GPU equal the oracle's merge of the same parts and the
    oracle's attention over all keys."""
    ensure_built()
    q, k, v = f32(*qkv_inputs.normal_qkv(2, 3, 5, 777, 64, seed=8))
    qd, kd, vd = (to_dev(x, torch.float32) for x in (q, k, v))
    po, pl = [], []
    for a, b in bounds:
        o, lse = pkg.attention(qd, kd[:, :, a:b].contiguous(), vd[:, :, a:b].contiguous())
        po.append(o.reshape(-1, 64))
        pl.append(lse.reshape(-1))
    po, pl = torch.stack(po), torch.stack(pl)
    om, lm = pkg.merge(po, pl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge_partials(po.double().cpu().numpy(), pl.double().cpu().numpy())
    om64 = om.double().cpu().numpy()
    if out_dtype == torch.float32:
        assert np.abs(om64 - o_ref).max() <= 1e-6
        full, full_lse = oracle.attention(q, k, v)
        assert np.abs(om64 - full.reshape(-1, 64)).max() <= 1e-5
        assert np.abs(lm.double().cpu().numpy() - full_lse.reshape(-1)).max() <= 1e-5
    else:
        assert_rounded_output(om64, o_ref, out_dtype)
    assert np.abs(lm.double().cpu().numpy() - lse_ref).max() <= 1e-5


def _sharded(qd, kd, vd, bounds, out_dtype):
    """Sequence-sharded attention as the bench's sharded workload runs it:
    each key shard contiguous (as on its own device), the tensor-core kernel
    on each with fp32 partial O and LSE, then attn_merge."""
    po, pl = [], []
    d = qd.shape[-1]
    for a, b in bounds:
        o, lse = pkg.attention(qd, kd[:, :, a:b].contiguous(), vd[:, :, a:b].contiguous(),
                               out_dtype=torch.float32)
        po.append(o.reshape(-1, d))
        pl.append(lse.reshape(-1))
    om, lm = pkg.merge(torch.stack(po), torch.stack(pl), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    return om, lm


@pytest.mark.parametrize("case", [
    # B, H, Sq, Skv, d, shard bounds
    (1, 4, 1024, 4096, 128, [(0, 1024), (1024, 2048), (2048, 3072), (3072, 4096)]),
    (2, 3, 300, 1000, 64, [(0, 333), (333, 666), (666, 1000)]),
    (1, 2, 129, 515, 128, [(0, 128), (128, 129), (129, 515)]),
])
def test_sequence_sharded_bf16_matches_oracle(case):
    """bf16 inputs, keys in contiguous shards (equal, unequal, one of a
    single key), the tensor-core kernel per shard, the merge to fp32 and to
    bf16 output: every row against the fp64 oracle over all keys, with the
    16-bit-input tolerances."""
    ensure_built()
    B, H, Sq, Skv, d, bounds = case
    q, k, v = qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=Skv + H, dtype=torch.bfloat16)
    o_ref, lse_ref = oracle.attention(q, k, v)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = o_ref.reshape(-1, d), lse_ref.reshape(-1)
    om, lm = _sharded(qd, kd, vd, bounds, torch.float32)
    assert_bf16_parity(om.double().cpu().numpy(), lm.double().cpu().numpy(), o_ref, lse_ref)
    ob, lb = _sharded(qd, kd, vd, bounds, torch.bfloat16)
    assert_rounded_output(ob.double().cpu().numpy(), o_ref, torch.bfloat16)
    assert torch.equal(lb, lm)


def test_sequence_sharded_b1_h32_s8192_sampled():
    """The bench's sharded workload at full size (B=1, H=32, Sq=Skv=8192,
    d=128, bf16, four shards of 2048 keys): every row finite; stratified rows
    of four heads against the oracle over all keys; and every row within the
    sum of both bounds of the unsharded attn_fwd."""
    ensure_built()
    B, H, S, d = 1, 32, 8192, 128
    q, k, v = qkv_inputs.normal_qkv(B, H, S, S, d, seed=0, dtype=torch.bfloat16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    bounds = [(i * 2048, (i + 1) * 2048) for i in range(4)]
    om, lm = _sharded(qd, kd, vd, bounds, torch.float32)
    assert torch.isfinite(om).all() and torch.isfinite(lm).all()
    o_whole, l_whole = pkg.attention(qd, kd, vd, out_dtype=torch.float32)
    torch.cuda.synchronize()
    # both are held to the oracle bounds, so they differ by at most their sum
    assert (om.reshape(B, H, S, d) - o_whole).abs().max().item() <= 2e-2
    assert (lm.reshape(B, H, S) - l_whole).abs().max().item() <= 2e-4 * max(
        1.0, l_whole.abs().max().item())
    qh, kh, vh = (t.reshape(B * H, S, d) for t in (q, k, v))
    omh = om.reshape(B * H, S, d).double().cpu().numpy()
    lmh = lm.reshape(B * H, S).double().cpu().numpy()
    got, got_l, refs, ref_l = [], [], [], []
    for bh in (0, 11, 22, 31):
        rs = qkv_inputs.sample_rows(S, 16, seed=2000 + bh)
        o_b, l_b = oracle.attention_rows(qh[bh:bh + 1], kh[bh:bh + 1], vh[bh:bh + 1],
                                         [(0, i) for i in rs])
        got.append(omh[bh, rs])
        got_l.append(lmh[bh, rs])
        refs.append(o_b)
        ref_l.append(l_b)
    assert_bf16_parity(np.concatenate(got), np.concatenate(got_l), np.concatenate(refs),
                       np.concatenate(ref_l))


def test_merge_empty_parts():
    ensure_built()
    po = torch.randn(3, 4, 32, device="cuda")
    pl = torch.tensor([[0.5, -math.inf, 1.0, -math.inf]] * 2 + [[-math.inf] * 4],
                      device="cuda")
    om, lm = pkg.merge(po, pl)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.merge_partials(po.double().cpu().numpy(), pl.double().cpu().numpy())
    assert np.abs(om.double().cpu().numpy() - o_ref).max() <= 1e-6
    assert torch.count_nonzero(om[1]).item() == 0 and torch.count_nonzero(om[3]).item() == 0
    assert math.isinf(lm[1].item()) and lm[1].item() < 0
    finite = np.isfinite(l_ref)
    assert np.abs(lm.double().cpu().numpy()[finite] - l_ref[finite]).max() <= 1e-6
