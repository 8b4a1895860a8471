"""Logical access model of aiml.sh "verify-tiled-attention" (function
``estimate_hbm_bytes``, section "Compare the attention outputs", and the
recorded ``hbm_traffic_sweep``).  TEST INFRASTRUCTURE ONLY.

It counts logical tensor accesses for one attention layer, not measured
traffic.  The dense method reads/writes Q, K, V, O once plus writes and reads
an N x N score matrix and an N x N probability matrix.  The causal tiled
loop reads Q and writes O once, and for every query block of ``block_q`` rows
re-reads K and V for all keys up to the end of that block, with no cache
reuse between blocks.  The caller's result is compared with the DRAM bytes a
profiler measures for the tiled GPU kernel.
"""
from __future__ import annotations

import math


def estimate_hbm_bytes(seq_len: int, num_heads: int = 32, head_dim: int = 128,
                       bytes_per_elem: int = 2, block_q: int = 128,
                       block_kv: int = 128) -> dict:
    """Logical bytes for dense and causal-tiled attention (see module doc).

    Values in MB are 1e6-byte units rounded to two decimals, as printed on
    the page; the exact byte counts are returned too."""
    del block_kv  # the page's model depends on the query block only
    per_tensor = num_heads * seq_len * head_dim * bytes_per_elem
    compulsory = 4 * per_tensor  # Q, K, V read + O written
    score_matrix_rw = 4 * num_heads * seq_len * seq_len * bytes_per_elem
    n_q_blocks = math.ceil(seq_len / block_q)
    # keys visible to the last row of each query block, summed over blocks
    kv_rows = sum(min(seq_len, start + block_q) for start in range(0, seq_len, block_q))
    tiled = (2 * per_tensor  # Q read + O written
             + 2 * num_heads * kv_rows * head_dim * bytes_per_elem)  # K and V
    return {
        "seq_len": seq_len,
        "num_heads": num_heads,
        "head_dim": head_dim,
        "num_q_blocks": n_q_blocks,
        "qkvo_compulsory_bytes": compulsory,
        "standard_nxn_matrix_bytes": score_matrix_rw,
        "standard_total_bytes": compulsory + score_matrix_rw,
        "tiled_logical_access_bytes": tiled,
        "qkvo_compulsory_bytes_mb": round(compulsory / 1e6, 2),
        "standard_nxn_matrix_hbm_mb": round(score_matrix_rw / 1e6, 2),
        "standard_total_hbm_mb": round((compulsory + score_matrix_rw) / 1e6, 2),
        "tiled_logical_access_mb_no_cache_reuse": round(tiled / 1e6, 2),
    }
