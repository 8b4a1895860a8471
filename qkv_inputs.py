"""Seeded synthetic Q/K/V generators shared by the oracle tests, the GPU parity
tests and the benchmark.

This module only draws random numbers and arranges them in the [B, H, S, d]
row-major layout; it contains none of the attention arithmetic.  Both the CUDA
path's tests and the oracle's tests take their inputs from here, so that the
two sides never share anything else.

Two families of inputs are produced:

* ``uniform`` -- the lab generator of aiml.sh "verify-tiled-attention"
  (``make_qkv``, section "Compare the attention outputs"): CPython
  ``random.Random(seed)``, values ``uniform(-0.8, 0.8)``, drawn for q first,
  then k, then v, each row-major.  For more than one (batch, head) pair the
  same stream continues, one (b, h) after another, q then k then v for each.
  With B = H = 1 and Sq = Skv this reproduces the page's ``make_qkv`` exactly.
* ``normal`` -- iid standard normal values from a seeded CPU
  ``torch.Generator`` (q, then k, then v, fp32), optionally rounded to bf16 or
  fp16 afterwards.  Used for the S=512 check of deepnotes
  "flash-attention-implemented-verified-and-measured" (section "Correctness
  first") and for the long-sequence bf16 workloads.
"""
from __future__ import annotations

import random

import numpy as np


def make_qkv(seq_len: int, head_dim: int, seed: int = 42):
    """Lists q, k, v of ``seq_len`` rows x ``head_dim`` values, drawn in the
    order of aiml.sh "verify-tiled-attention" (``make_qkv``)."""
    rng = random.Random(seed)
    q = [[rng.uniform(-0.8, 0.8) for _ in range(head_dim)] for _ in range(seq_len)]
    k = [[rng.uniform(-0.8, 0.8) for _ in range(head_dim)] for _ in range(seq_len)]
    v = [[rng.uniform(-0.8, 0.8) for _ in range(head_dim)] for _ in range(seq_len)]
    return q, k, v


def uniform_qkv(B: int, H: int, Sq: int, Skv: int, d: int, seed: int,
                low: float = -0.8, high: float = 0.8):
    """fp64 numpy arrays q [B,H,Sq,d], k and v [B,H,Skv,d] from one
    ``random.Random(seed)`` stream, (b, h) pairs in order, q then k then v."""
    rng = random.Random(seed)
    q = np.empty((B, H, Sq, d), dtype=np.float64)
    k = np.empty((B, H, Skv, d), dtype=np.float64)
    v = np.empty((B, H, Skv, d), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for arr, rows in ((q, Sq), (k, Skv), (v, Skv)):
                flat = [rng.uniform(low, high) for _ in range(rows * d)]
                arr[b, h] = np.asarray(flat, dtype=np.float64).reshape(rows, d)
    return q, k, v


def normal_qkv(B: int, H: int, Sq: int, Skv: int, d: int, seed: int,
               dtype=None):
    """CPU torch tensors q [B,H,Sq,d], k and v [B,H,Skv,d]: iid standard
    normal fp32 from ``torch.Generator().manual_seed(seed)`` (q, k, v in that
    order), then cast to ``dtype`` (round to nearest even) when given."""
    import torch

    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, H, Sq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Skv, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Skv, d), generator=g, dtype=torch.float32)
    if dtype is not None and dtype != torch.float32:
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    return q, k, v


def normal_qkv_device(B: int, H: int, Sq: int, Skv: int, d: int, seed: int,
                      dtype, device):
    """Same distribution as :func:`normal_qkv`, drawn directly on ``device``
    from a seeded device generator (used where only the distribution matters,
    e.g. timing; parity tests use the CPU generator)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for S in (Sq, Skv, Skv):
        t = torch.randn((B, H, S, d), generator=g, dtype=torch.float32, device=device)
        out.append(t.to(dtype))
    return tuple(out)


def sample_rows(Sq: int, n_random: int, seed: int, tile: int = 128):
    """Fixed stratified set of query-row indices used for sampled parity on
    workloads too large for the fp64 oracle: the first four rows, the rows on
    either side of every ``tile`` boundary, the last four rows, and
    ``n_random`` seeded uniform rows.  Sorted, unique, all < Sq."""
    rows = set(range(min(4, Sq)))
    for b in range(tile, Sq, tile):
        rows.add(b - 1)
        rows.add(b)
    rows.update(range(max(0, Sq - 4), Sq))
    rng = random.Random(seed)
    for _ in range(n_random):
        rows.add(rng.randrange(Sq))
    return sorted(rows)
