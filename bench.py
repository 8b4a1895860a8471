"""Benchmark: exact attention forward on GB300, TFLOP/s and fraction of the
dense bf16 tensor-core peak.

Default workload: B=1, H=32, Sq=Skv=8192, d=128, bf16 inputs with fp32
accumulation, causal, scale 1/sqrt(128), iid standard-normal Q/K/V (seeded).
A step is one attn_fwd launch over that batch.  Work per step is
4*B*H*Sq*Skv*d FLOP, halved for causal.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl reference]

Prints one JSON line.  For N > 1 run it under torch.distributed.run: every
rank processes its own batch on its own GPU (no collective on the data path),
timing is the maximum over ranks, and ``value`` counts the work of all ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s at 1 GB300 (bf16, causal) and % of dense bf16 tensor peak"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2

CONFIGS = {
    # name: (B, H, Sq, Skv, d, causal, dtype, input family)
    "b1_h1_s64_d32_f32": (1, 1, 64, 64, 32, True, "f32", "uniform"),
    "b1_h1_q8_kv1024_d32_f32": (1, 1, 8, 1024, 32, False, "f32", "uniform"),
    "b2_h4_s512_d64_f32": (2, 4, 512, 512, 64, False, "f32", "normal"),
    "b1_h32_s8192_d128_bf16_causal": (1, 32, 8192, 8192, 128, True, "bf16", "normal"),
    "b1_h64_s32768_d128_bf16_causal": (1, 64, 32768, 32768, 128, True, "bf16", "normal"),
    # decode: one query row per head against a long key sequence, split-KV path
    "b4_h32_q1_kv32768_d128_bf16_decode": (4, 32, 1, 32768, 128, False, "bf16", "normal"),
    # the access-model sweep of aiml.sh "verify-tiled-attention" (H=32, d=128, causal)
    "b1_h32_s1024_d128_bf16_causal": (1, 32, 1024, 1024, 128, True, "bf16", "normal"),
    "b1_h32_s4096_d128_bf16_causal": (1, 32, 4096, 4096, 128, True, "bf16", "normal"),
    "b1_h32_s16384_d128_bf16_causal": (1, 32, 16384, 16384, 128, True, "bf16", "normal"),
    "b1_h32_s32768_d128_bf16_causal": (1, 32, 32768, 32768, 128, True, "bf16", "normal"),
    # other variants of the tensor-core kernel
    "b1_h32_s8192_d128_fp16_causal": (1, 32, 8192, 8192, 128, True, "f16", "normal"),
    "b1_h64_s8192_d64_bf16_causal": (1, 64, 8192, 8192, 64, True, "bf16", "normal"),
    "b1_h32_s8192_d128_bf16_full": (1, 32, 8192, 8192, 128, False, "bf16", "normal"),
    # sequence-sharded: the keys in 4 contiguous shards, as separate devices would hold
    # them; attn_fwd on each shard (fp32 partial O and LSE), then attn_merge
    "b1_h32_s8192_d128_bf16_full_kv4shards": (1, 32, 8192, 8192, 128, False, "bf16", "normal"),
}
# few query rows against many keys: the split-KV path (partial kernel + merge)
SPLITKV = {"b4_h32_q1_kv32768_d128_bf16_decode", "b1_h1_q8_kv1024_d32_f32"}
# sequence-sharded workloads: number of key shards (non-causal only: a causal mask
# does not split into per-shard bottom-right masks)
SHARDED = {"b1_h32_s8192_d128_bf16_full_kv4shards": 4}
# fp32 workloads whose arithmetic, not their bytes, bounds them (about 128 FLOP per byte)
FP32_ALU = {"b2_h4_s512_d64_f32"}
FP32_FMA_PER_CLK_PER_SM = 128  # CUDA-core FP32 lanes of one SM
DEFAULT = "b1_h32_s8192_d128_bf16_causal"


def compulsory_bytes(cfg):
    """Bytes every implementation must move: Q, K, V read, O and LSE written."""
    B, H, Sq, Skv, d, causal, dt, _ = cfg
    e = 4 if dt == "f32" else 2
    return B * H * (Sq * d * e * 2 + 2 * Skv * d * e + Sq * 4)


def flops(B, H, Sq, Skv, d, causal):
    f = 4.0 * B * H * Sq * Skv * d
    return f / 2 if causal else f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def kernel_source_hash(config_name=DEFAULT):
    """Hash of the source files of the dominant kernel of a workload."""
    if config_name in SPLITKV:
        files = ("attn_splitkv.cu",)
    elif CONFIGS[config_name][6] == "f32":
        files = ("attn_f32.cu",)
    else:
        files = ("attn_tc.cu", "sm100_ptx.cuh")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "online_softmax_forward_gb300", "csrc", f)) as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def code_only(src):
    """CUDA/C++ source with comments removed and whitespace collapsed, so that
    an edit of comments alone keeps the kernel's hash."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def profiled_traffic(config_name):
    """DRAM bytes per launch recorded from an ncu capture of this kernel
    source (profiles/*.md line 'traffic_bytes_per_launch: N kernel_sha: H
    config: C'); None if absent or taken on another kernel version."""
    pdir = os.path.join(ROOT, "profiles")
    want = kernel_source_hash(config_name)
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(r"traffic_bytes_per_launch:\s*(\d+)\s+kernel_sha:\s*(\w+)\s+config:\s*(\S+)")
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith(".md"):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(2) == want and m.group(3) == config_name:
                    return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def make_inputs(cfg, device, seed=0):
    import torch
    import qkv_inputs
    B, H, Sq, Skv, d, causal, dt, family = cfg
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dt]
    if family == "uniform":
        q, k, v = (torch.from_numpy(a) for a in qkv_inputs.uniform_qkv(B, H, Sq, Skv, d, 42))
        return tuple(t.to(tdt).to(device) for t in (q, k, v))
    return qkv_inputs.normal_qkv_device(B, H, Sq, Skv, d, seed, tdt, device)


def dtype_code(cfg):
    import online_softmax_forward_gb300 as pkg
    return {"f32": pkg.ATTN_F32, "bf16": pkg.ATTN_BF16, "f16": pkg.ATTN_F16}[cfg[6]]


# ------------------------------------------------------------------ our arm
def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import online_softmax_forward_gb300 as pkg
    from online_softmax_forward_gb300 import build as lib_build

    if rank == 0 or not os.path.exists(pkg.library_path()):
        lib_build.build()
    if world > 1:
        dist.barrier()
    pkg.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = CONFIGS[args.config]
    B, H, Sq, Skv, d, causal, dt, _ = cfg
    code = dtype_code(cfg)
    q, k, v = make_inputs(cfg, dev, seed=rank)
    odt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dt]
    o = torch.empty((B, H, Sq, d), dtype=odt, device=dev)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    splitkv = args.config in SPLITKV
    n_shards = SHARDED.get(args.config, 0)
    if n_shards:
        # each shard contiguous, as on its own device; fp32 partials [n, B, H, Sq, (d)]
        sk = Skv // n_shards
        k_sh = [k[:, :, i * sk:(i + 1) * sk].contiguous() for i in range(n_shards)]
        v_sh = [v[:, :, i * sk:(i + 1) * sk].contiguous() for i in range(n_shards)]
        o_parts = torch.empty((n_shards, B, H, Sq, d), dtype=torch.float32, device=dev)
        lse_parts = torch.empty((n_shards, B, H, Sq), dtype=torch.float32, device=dev)
        part_code = {"bf16": pkg.ATTN_BF16_OUT_F32, "f16": pkg.ATTN_F16_OUT_F32,
                     "f32": pkg.ATTN_F32}[dt]
    n_splits, ws = 0, None
    if splitkv:
        st, n_splits, ws_bytes = pkg.attn_splitkv_plan(B, H, Sq, Skv, d, code)
        if st != pkg.ATTN_OK:
            raise pkg.AttnError(st, "attn_splitkv_plan")
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def launch_sharded(qq, ks, vs, mark=None):
        for i in range(n_shards):
            st = pkg.attn_fwd(qq.data_ptr(), ks[i].data_ptr(), vs[i].data_ptr(),
                              o_parts[i].data_ptr(), lse_parts[i].data_ptr(), B, H, Sq, sk, d,
                              0, 0.0, part_code, sh)
            if st != pkg.ATTN_OK:
                raise pkg.AttnError(st, "attn_fwd (shard)")
        if mark is not None:
            mark.record(stream)  # the shards' kernels end here, the merge follows
        st = pkg.attn_merge(o_parts.data_ptr(), lse_parts.data_ptr(), n_shards, B * H * Sq, d,
                            o.data_ptr(), lse.data_ptr(), code, sh)
        if st != pkg.ATTN_OK:
            raise pkg.AttnError(st, "attn_merge")

    def launch(qq=q, kk=k, vv=v, mark=None):
        if n_shards:
            launch_sharded(qq, k_sh if kk is k else kk, v_sh if vv is v else vv, mark)
            return
        if splitkv:
            st = pkg.attn_fwd_splitkv(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code,
                                      n_splits, ws.data_ptr(), ws.numel(), sh)
        else:
            st = pkg.attn_fwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0, code, sh)
        if st != pkg.ATTN_OK:
            raise pkg.AttnError(st, "attn_fwd_splitkv" if splitkv else "attn_fwd")

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            launch()
        stream.synchronize()
        assert pkg.attn_check_status(sh) == pkg.ATTN_OK

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if n_shards else None
        sampler = ClockSampler(local_rank)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler.start()
        time.sleep(0.3)  # let the sampler take its first reading
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)          # evict L2 between steps (outside the events)
            starts[i].record(stream)
            launch(mark=mids[i] if n_shards else None)
            ends[i].record(stream)
        stream.synchronize()
        wall = time.perf_counter() - t_wall
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clocks = sampler.stop()
        st = pkg.attn_check_status(sh)
        if st != pkg.ATTN_OK:
            raise pkg.AttnError(st, "attn_check_status")
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms per launch
    # sequence-sharded: the time of the shards' tensor-core kernels alone, for the
    # roofline of that (dominant) kernel; the merge follows in the step
    shard_ms = (sum(s.elapsed_time(m) for s, m in zip(starts, mids)) / len(mids)
                if n_shards else None)
    ms = sum(times) / len(times)

    # e2e: host buffers through attn_fwd_staged, copies inside the timed region
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    if n_shards:
        kh_sh = [t.cpu().pin_memory() for t in k_sh]
        vh_sh = [t.cpu().pin_memory() for t in v_sh]
        dk_sh = [torch.empty_like(t) for t in k_sh]
        dv_sh = [torch.empty_like(t) for t in v_sh]
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    e2e_times = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            stream.synchronize()
            t0 = time.perf_counter()
            if n_shards:  # host -> device copies of q and every shard, the shards, the merge
                dq.copy_(qh, non_blocking=True)
                for dst, src_ in zip(dk_sh + dv_sh, kh_sh + vh_sh):
                    dst.copy_(src_, non_blocking=True)
                launch(dq, dk_sh, dv_sh)
                oh.copy_(o, non_blocking=True)
                lh.copy_(lse, non_blocking=True)
            elif splitkv:  # host -> device copies, the split-KV call, device -> host copies
                for dst, src_ in ((dq, qh), (dk, kh), (dv, vh)):
                    dst.copy_(src_, non_blocking=True)
                launch(dq, dk, dv)
                oh.copy_(o, non_blocking=True)
                lh.copy_(lse, non_blocking=True)
            else:
                st = pkg.attn_fwd_staged(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(),
                                         oh.data_ptr(), lh.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, H, Sq, Skv, d, int(causal), 0.0,
                                         code, sh)
                if st != pkg.ATTN_OK:
                    raise pkg.AttnError(st, "attn_fwd_staged")
            stream.synchronize()
            if i >= args.warmup:
                e2e_times.append(time.perf_counter() - t0)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = o.numel() * o.element_size() + lse.numel() * 4

    f = flops(B, H, Sq, Skv, d, causal)
    # max over ranks of the per-step device time
    ms_max, e2e_s, shard_max = max_over_ranks(
        [ms, sum(e2e_times) / len(e2e_times), shard_ms if n_shards else 0.0], world, dev)
    return dict(ms=ms_max, flops=f, times=times, wall=wall, clocks=clocks, e2e_s=e2e_s,
                h2d=h2d, d2h=d2h, cfg=cfg,
                launches_per_step=n_shards + 1 if n_shards else (2 if splitkv else 1),
                n_splits=n_splits, shard_ms=shard_max if n_shards else None)


def cpu_baseline(cfg, target_s=12.0):
    """The fp64 oracle on a bounded sample of rows of the same workload, on
    all host cores; returns TFLOP/s counted like the GPU metric."""
    import numpy as np
    import torch

    import oracle
    import qkv_inputs
    B, H, Sq, Skv, d, causal, dt, family = cfg
    if family == "uniform":
        q, k, v = (torch.from_numpy(a) for a in qkv_inputs.uniform_qkv(B, H, Sq, Skv, d, 42))
    else:
        # the heads sampled below only: draw the full tensors for the first head
        q, k, v = qkv_inputs.normal_qkv(1, 1, Sq, Skv, d, 0,
                                        dtype={"bf16": torch.bfloat16,
                                               "f16": torch.float16}.get(dt))
    qh, kh, vh = (t.reshape(-1, t.shape[-2], d)[:1] for t in (q, k, v))
    off = Skv - Sq
    nthreads = os.cpu_count() or 1

    def row_flops(i):
        n = min(Skv, max(0, i + 1 + off)) if causal else Skv
        return 4.0 * n * d

    def timed(rows):
        t0 = time.perf_counter()
        oracle.attention_rows(qh, kh, vh, [(0, i) for i in rows], causal=causal,
                              nthreads=nthreads)
        return time.perf_counter() - t0

    # calibrate on a small stratified sample, then size the main sample
    stride = max(1, Sq // 64)
    probe = list(range(0, Sq, stride))
    t_probe = timed(probe)
    f_probe = sum(row_flops(i) for i in probe)
    rate = f_probe / max(t_probe, 1e-6)
    want_rows = int(target_s * rate / (sum(row_flops(i) for i in range(Sq)) / Sq))
    want_rows = max(len(probe), min(Sq * B * H, want_rows))
    stride = max(1, Sq // max(1, min(Sq, want_rows)))
    rows = list(range(0, Sq, stride))
    reps = max(1, want_rows // max(1, len(rows)))
    t = 0.0
    fl = 0.0
    for _ in range(reps):
        t += timed(rows)
        fl += sum(row_flops(i) for i in rows)
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d query rows (every %d-th row of one head, %d pass(es)) of the same "
                      "workload, fp64 dense per-row oracle, %.1f s" % (len(rows), stride, reps, t),
            "seconds": t, "flops": fl}


def max_over_ranks(values, world, device):
    """Element-wise maximum of a list of floats over all ranks (identity for a
    single process)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local_rank


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = init_dist()
    cfg = CONFIGS[args.config]
    B, H, Sq, Skv, d, causal, dt, _ = cfg
    peaks = load_peaks()
    config = {"workload": args.config, "B": B, "H": H, "Sq": Sq, "Skv": Skv, "d": d,
              "path": ("split-KV (attn_fwd_splitkv)" if args.config in SPLITKV else
                       "sequence-sharded: attn_fwd on %d key shards (fp32 partials) + attn_merge"
                       % SHARDED[args.config] if args.config in SHARDED else "attn_fwd"),
              "causal": causal, "inputs": "iid standard normal, seeded" if cfg[7] == "normal"
              else "iid uniform(-0.8,0.8), random.Random(42)",
              "l2": "flushed between steps (256 MiB fill outside the kernel events)",
              "per_rank_batch": "B*H heads per GPU"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        res = [cpu_baseline(cfg, target_s=max(3.0, 12.0 / max(1, args.steps)))
               for _ in range(args.warmup + args.steps)][args.warmup:]
        vals = [r["value"] for r in res]
        v = statistics.median(vals)
        line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": statistics.median(r["seconds"] for r in res) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": config, "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "kind": "oracle",
                                 "cores": res[0]["cores"], "sample": res[0]["sample"]},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line))
        return 0

    r = run_gpu(args, rank, world, local_rank)
    if rank != 0:
        return 0
    tflops = r["flops"] / (r["ms"] * 1e-3) / 1e12
    value = world * tflops
    if cfg[6] in ("bf16", "f16") and args.config not in SPLITKV:
        # fp16 and bf16 share the dense tensor-core rate: the bf16 measured peak serves both
        peak, unit, bound = peaks["bf16_tflops"], "TFLOP/s", "tensor"
        achieved = tflops
        peak_source = peaks["source"] + " burst bf16 (kernel timed alone)"
        if r["shard_ms"]:
            # the dominant kernel: the shards' tensor-core launches, without the merge
            achieved = r["flops"] / (r["shard_ms"] * 1e-3) / 1e12
            peak_source += "; achieved over the shard kernels' time, merge excluded"
    elif args.config in FP32_ALU:
        # FP32 FMA rate from the unit count and the maximum SM clock
        import torch
        sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
        mhz = (r["clocks"] or {}).get("sm_max_mhz") or 2070.0
        peak = sms * FP32_FMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12
        unit, bound, achieved = "TFLOP/s", "alu", tflops
        peak_source = "derived: %d SMs x %d FP32 FMA/clk x 2 FLOP x %.0f MHz" % (
            sms, FP32_FMA_PER_CLK_PER_SM, mhz)
    else:
        # decode and the small fp32 cases: compulsory bytes against HBM
        peak, unit, bound = peaks["hbm_gbs"], "GB/s", "hbm"
        achieved = compulsory_bytes(cfg) / (r["ms"] * 1e-3) / 1e9
        peak_source = peaks["source"] + " copy GB/s"
    traffic = profiled_traffic(args.config)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dt, "data": "synthetic", "config": config,
        "pct_of_dense_bf16_peak": (100.0 * tflops / peaks["bf16_tflops"]
                                   if dt in ("bf16", "f16") else None),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_source},
        "e2e": {"value": world * r["flops"] / r["e2e_s"] / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": args.steps * r["launches_per_step"],
        "clocks": r["clocks"],
        "step_ms_min": min(r["times"]), "step_ms_max": max(r["times"]),
    }
    if world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(cfg)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
