"""The dynamic schedule of the tensor-core kernel: every launch takes its work
units from one of 256 device counter pairs, in turn, and its last CTA returns
the pair to zero.  A pair that was not returned to zero would make a later
launch on it skip units, leaving parts of its output unwritten.

These tests make many launches -- more than two full turns over the counters,
on two streams with nothing ordering them, so launches on different counters
run concurrently -- into outputs pre-filled with NaN, and require every
output to equal, bit for bit, the output of a single reference call."""
import pytest
import torch

import online_softmax_forward_gb300 as pkg
import qkv_inputs
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


def _problem():
    B, H, S, d = 1, 3, 700, 128  # ragged: 700 = 5 * 128 + 60; 9 units
    q, k, v = (t.cuda() for t in qkv_inputs.normal_qkv(B, H, S, S, d, seed=51,
                                                       dtype=torch.bfloat16))
    return q, k, v


def test_counters_wrap_and_reset_across_streams():
    ensure_built()
    q, k, v = _problem()
    ref_o, ref_l = pkg.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    n = 600  # more than twice the 256 counter pairs
    outs = [(torch.full_like(ref_o, float("nan")), torch.full_like(ref_l, float("nan")))
            for _ in range(n)]
    torch.cuda.synchronize()
    for i, (o, lse) in enumerate(outs):
        pkg.attention(q, k, v, causal=True, out=o, lse=lse, stream=streams[i & 1])
    torch.cuda.synchronize()
    for s in streams:
        assert pkg.attn_check_status(s.cuda_stream) == pkg.ATTN_OK
    bad = [i for i, (o, lse) in enumerate(outs) if not (torch.equal(o, ref_o) and torch.equal(lse, ref_l))]
    assert not bad, "outputs differing from the reference: %s" % bad[:10]


def test_aborted_launch_returns_its_counter():
    """On the test library (the only one with the watchdog hook): a launch
    stopped by an expired wait still returns its counter pair to zero, so
    the launch that reuses the pair 256 calls later is complete."""
    ensure_built()
    tl = pkg.load_test_library()
    q, k, v = _problem()
    B, H, S, d = q.shape
    ref_o, ref_l = pkg.attention(q, k, v, causal=True)
    torch.cuda.synchronize()

    def fwd(o, lse):
        st = tl.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, H, S, S, d, 1, 0.0, pkg.ATTN_BF16, None)
        assert st == pkg.ATTN_OK

    scratch = (torch.empty_like(ref_o), torch.empty_like(ref_l))
    try:
        assert tl.attn_test_set_hook(1, 20_000_000) == pkg.ATTN_OK
        fwd(*scratch)  # gives up a wait: its output is incomplete
        assert tl.attn_check_status(None) == pkg.ATTN_ERR_TIMEOUT
    finally:
        assert tl.attn_test_set_hook(0, 1_000_000_000) == pkg.ATTN_OK
    outs = [(torch.full_like(ref_o, float("nan")), torch.full_like(ref_l, float("nan")))
            for _ in range(257)]
    for o, lse in outs:  # the last one takes the aborted launch's counter pair again
        fwd(o, lse)
    torch.cuda.synchronize()
    assert tl.attn_check_status(None) == pkg.ATTN_OK
    for o, lse in outs:
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_concurrent_host_threads():
    """Four host threads call the library at the same time, each on its own
    stream and with its own outputs (the calls release the interpreter lock):
    the per-device caches, the choice of counter pairs and the kernels running
    side by side must not disturb one another."""
    import threading
    ensure_built()
    q, k, v = _problem()
    ref_o, ref_l = pkg.attention(q, k, v, causal=True)
    qf, kf, vf = (t.float() for t in (q[:, :1, :200, :64], k[:, :1, :200, :64], v[:, :1, :200, :64]))
    qf, kf, vf = (t.contiguous() for t in (qf, kf, vf))
    ref_f, _ = pkg.attention(qf, kf, vf, causal=True)
    torch.cuda.synchronize()
    n_threads, n_calls = 4, 40
    outs = [[(torch.full_like(ref_o, float("nan")), torch.full_like(ref_l, float("nan")),
              torch.full_like(ref_f, float("nan"))) for _ in range(n_calls)]
            for _ in range(n_threads)]
    streams = [torch.cuda.Stream() for _ in range(n_threads)]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(q.device)
            for o, lse, of in outs[i]:
                pkg.attention(q, k, v, causal=True, out=o, lse=lse, stream=streams[i])
                pkg.attention(qf, kf, vf, causal=True, out=of, return_lse=False,
                              stream=streams[i])
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for s in streams:
        assert pkg.attn_check_status(s.cuda_stream) == pkg.ATTN_OK
    for i in range(n_threads):
        for o, lse, of in outs[i]:
            assert torch.equal(o, ref_o) and torch.equal(lse, ref_l) and torch.equal(of, ref_f)


def test_full_size_launches_identical():
    """B=1, H=32, S=8192, d=128 causal (1,024 units over the persistent grid,
    several claims per CTA): 40 launches, each into an output pre-filled with
    NaN, must each equal the first launch bit for bit -- the units a CTA
    claims differ from launch to launch, the result may not."""
    ensure_built()
    q, k, v = (t.cuda() for t in qkv_inputs.normal_qkv(1, 32, 8192, 8192, 128, seed=52,
                                                       dtype=torch.bfloat16))
    ref_o, ref_l = pkg.attention(q, k, v, causal=True)
    torch.cuda.synchronize()
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    bad = 0
    for _ in range(40):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        pkg.attention(q, k, v, causal=True, out=o, lse=lse)
        bad += int(not (torch.equal(o, ref_o) and torch.equal(lse, ref_l)))
    torch.cuda.synchronize()
    assert pkg.attn_check_status(None) == pkg.ATTN_OK
    assert bad == 0
