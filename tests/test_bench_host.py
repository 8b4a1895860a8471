"""Host-side logic of bench.py: FLOP convention, the max-over-ranks timing of
a multi-process run (gloo, world size 2, CPU), and the reference arm's
rank-0-only output under torch.distributed.run."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_flop_convention():
    # 4*B*H*Sq*Skv*d, halved for causal
    assert bench.flops(1, 32, 8192, 8192, 128, True) == 4 * 32 * 8192 * 8192 * 128 / 2
    assert bench.flops(2, 4, 512, 512, 64, False) == 4 * 2 * 4 * 512 * 512 * 64
    assert abs(bench.flops(1, 32, 8192, 8192, 128, True) - 5.498e11) / 5.498e11 < 1e-3


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world, torch.device("cpu"))
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, BENCH_BACKEND="gloo")
    port = 30500 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--config", "b1_h1_s64_d32_f32"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s"
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_compulsory_bytes_and_paths():
    # decode: q, o (bf16), k, v (bf16) and lse (fp32)
    cfg = bench.CONFIGS["b4_h32_q1_kv32768_d128_bf16_decode"]
    B, H, Sq, Skv, d = 4, 32, 1, 32768, 128
    assert bench.compulsory_bytes(cfg) == B * H * (2 * Sq * d * 2 + 2 * Skv * d * 2 + Sq * 4)
    assert "b4_h32_q1_kv32768_d128_bf16_decode" in bench.SPLITKV
    assert bench.DEFAULT not in bench.SPLITKV
    # the traffic record is keyed by the source of the workload's dominant kernel
    assert bench.kernel_source_hash(bench.DEFAULT) != \
        bench.kernel_source_hash("b4_h32_q1_kv32768_d128_bf16_decode")


def test_kernel_hash_ignores_comments_only():
    a = "int f(int x) {  // one\n  return x + 1; /* two */ }\n"
    b = "/* header */\nint f(int x) {\n  return x + 1;\n}  // trailing\n"
    c = "int f(int x) { return x + 2; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)


def test_sharded_workloads_split_evenly_and_are_not_causal():
    """A bottom-right causal mask does not split into per-shard masks, and
    the bench cuts the keys into equal contiguous shards."""
    assert bench.SHARDED
    for name, n in bench.SHARDED.items():
        B, H, Sq, Skv, d, causal, dt, _ = bench.CONFIGS[name]
        assert not causal and n >= 2 and Skv % n == 0
        assert name not in bench.SPLITKV
        # the dominant kernel is the tensor-core kernel of the shards
        assert bench.kernel_source_hash(name) == bench.kernel_source_hash(bench.DEFAULT)
