"""attn_fwd and attn_fwd_splitkv inside a CUDA graph.

After one ordinary call, which sets up the per-device kernel attributes and the
status word, each path is captured with torch.cuda.graph and replayed on new
input values copied into the captured input tensors. Every replay must equal
an ordinary call on the same inputs bit for bit. The paths covered are the
tensor-core kernel, the fp32 kernel and split-KV with its merge.

A serving loop relies on this: nothing in these calls allocates, synchronises
or reads host state that would be frozen into the graph, apart from the
problem shape."""
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import qkv_inputs
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Sq, Skv, d, causal, dtype, path
    (1, 4, 600, 600, 128, True, torch.bfloat16, "fwd"),
    (1, 2, 300, 517, 64, False, torch.float16, "fwd"),
    (2, 3, 130, 300, 64, False, torch.float32, "fwd"),
    (2, 4, 1, 5000, 128, False, torch.bfloat16, "splitkv"),
    (1, 2, 9, 777, 64, True, torch.float32, "splitkv"),
]


@pytest.mark.parametrize("case", CASES)
def test_graph_replay_matches_direct_call(case):
    ensure_built()
    B, H, Sq, Skv, d, causal, dt, path = case

    def call(q, k, v):
        if path == "fwd":
            return pkg.attention(q, k, v, causal=causal)
        return pkg.attention_splitkv(q, k, v, causal=causal)

    inputs = [[t.to(dt).cuda() for t in qkv_inputs.normal_qkv(B, H, Sq, Skv, d, seed=s)]
              for s in (11, 12, 13)]
    sq, sk, sv = (t.clone() for t in inputs[0])
    call(sq, sk, sv)  # set-up happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        go, gl = call(sq, sk, sv)
    for q, k, v in inputs[1:] + inputs[:1]:
        sq.copy_(q)
        sk.copy_(k)
        sv.copy_(v)
        g.replay()
        o, lse = call(q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(go, o) and torch.equal(gl, lse)
    assert pkg.attn_check_status(None) == pkg.ATTN_OK


def test_wrappers_refuse_mismatched_outputs_before_launching():
    """Caller-provided outputs and workspaces are checked against what the
    call writes (shape, dtype, contiguity, device) on the host: a mismatch is
    a ValueError and the output stays untouched."""
    ensure_built()
    q, k, v = (t.to(torch.bfloat16).cuda() for t in qkv_inputs.normal_qkv(1, 2, 64, 64, 64, seed=5))
    bad_shape = torch.full((1, 2, 63, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    bad_dtype = torch.full((1, 2, 64, 64), 7.0, dtype=torch.float16, device="cuda")
    strided = torch.full((1, 2, 64, 128), 7.0, dtype=torch.bfloat16, device="cuda")[..., ::2]
    host = torch.full((1, 2, 64, 64), 7.0, dtype=torch.bfloat16)
    for out in (bad_shape, bad_dtype, strided, host):
        with pytest.raises(ValueError):
            pkg.attention(q, k, v, out=out)
        assert torch.all(out == 7.0)
    with pytest.raises(ValueError):
        pkg.attention(q, k, v, lse=torch.zeros((1, 2, 64), dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        pkg.attention_splitkv(q, k, v, n_splits=2, workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
