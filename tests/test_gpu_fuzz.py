"""Seeded random shapes through every path, each compared element by element
with the fp64 oracle.  The shapes are drawn once from a fixed seed, so the
cases are the same on every run: B, H in 1..3, Sq and Skv in 1..700 (ragged
against every tile size the kernels use) and, for ten more, in 1..3000, causal or not, every supported
head width and input type, fp32 or 16-bit output, attn_fwd and split-KV with
a random split count."""
import random

import pytest
import torch

import online_softmax_forward_gb300 as pkg
import oracle
import qkv_inputs
from gpu_util import (assert_bf16_parity, assert_f32_parity, assert_lse_close,
                      assert_rounded_output, ensure_built)

pytestmark = pytest.mark.gpu


def _cases(n, seed, max_len=700, first=0):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        dt = rng.choice([torch.float32, torch.bfloat16, torch.float16])
        d = rng.choice([16, 32, 64, 128] if dt == torch.float32 else [64, 128])
        out.append(dict(
            B=rng.randint(1, 3), H=rng.randint(1, 3), Sq=rng.randint(1, max_len),
            Skv=rng.randint(1, max_len), d=d, causal=rng.random() < 0.5, dtype=dt,
            out32=dt == torch.float32 or rng.random() < 0.5,
            splitkv=rng.random() < 0.3, n_splits=rng.randint(1, 12), seed=1000 + first + i))
    return out


# short sequences (every tile size, ragged), then longer ones (several units per
# head on the tensor-core kernel, several key tiles per warp on the fp32 kernels)
CASES = _cases(24, 20261203) + _cases(10, 7, max_len=3000, first=100)


def _id(c):
    return "%s_B%dH%d_%dx%d_d%d_%s%s%s" % (
        str(c["dtype"]).split(".")[-1], c["B"], c["H"], c["Sq"], c["Skv"], c["d"],
        "causal" if c["causal"] else "full", "_o32" if c["out32"] else "",
        "_splitkv%d" % c["n_splits"] if c["splitkv"] else "")


@pytest.mark.parametrize("c", CASES, ids=_id)
def test_random_shape_matches_oracle(c):
    ensure_built()
    B, H, Sq, Skv, d = c["B"], c["H"], c["Sq"], c["Skv"], c["d"]
    dt, causal = c["dtype"], c["causal"]
    q, k, v = (t.to(dt) for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=c["seed"]))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    odt = torch.float32 if c["out32"] else dt
    if c["splitkv"]:
        o, lse = pkg.attention_splitkv(qd, kd, vd, causal=causal, out_dtype=odt,
                                       n_splits=c["n_splits"])
    else:
        o, lse = pkg.attention(qd, kd, vd, causal=causal, out_dtype=odt)
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    o, lse = o.double().cpu().numpy(), lse.double().cpu().numpy()
    if dt == torch.float32:
        assert_f32_parity(o, lse, o_ref, lse_ref)
    elif c["out32"]:
        assert_bf16_parity(o, lse, o_ref, lse_ref)
    else:
        assert_rounded_output(o, o_ref, dt)
        assert_lse_close(lse, lse_ref, 1e-4)
