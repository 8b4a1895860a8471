"""O2: the tiled online-softmax algorithm restated in fp64 NumPy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is not the parity
oracle -- ``oracle.attention`` is.  It exists to test the *algorithm*: that
the result does not depend on the tile sizes, that omitting the accumulator
rescale breaks it, and that the worked example of the pages comes out right.

The steps follow aiml.sh "verify-tiled-attention" (``tiled_flash_attention``:
an outer loop over query blocks, an inner loop over key/value blocks that
stops at the first block lying wholly past the causal limit, a per-row set of
visible keys, and per-row running maximum / normaliser / accumulator), with
the update written in the notation of huhohoo "tiled-online-softmax"
("Online normalization"):

    m_new = max(m, max(S))
    rescale = exp(m - m_new)            (0 while m is still -inf)
    P = exp(S - m_new)
    a = a * rescale + P @ V_block
    l = l * rescale + sum(P)
    output = a / l

The rows of one query block are processed together as vectors; a row with no
visible key in a tile leaves its state untouched, which is what the page's
per-row ``continue`` does.
"""
from __future__ import annotations

import math

import numpy as np


def _one_head(q, k, v, block_q, block_kv, causal, scale, rescale_previous_acc):
    sq, d = q.shape
    skv = k.shape[0]
    offset = skv - sq  # bottom-right causal alignment; 0 on the pages
    out = np.zeros((sq, d), dtype=np.float64)
    lse = np.full((sq,), -math.inf, dtype=np.float64)
    tiles_visited = 0
    for q_start in range(0, sq, block_q):
        q_end = min(q_start + block_q, sq)
        rows = np.arange(q_start, q_end)
        m = np.full((q_end - q_start,), -math.inf)
        l = np.zeros((q_end - q_start,))
        a = np.zeros((q_end - q_start, d))
        for kv_start in range(0, skv, block_kv):
            # the last row of the block sees keys j <= (q_end - 1) + offset
            if causal and kv_start > q_end - 1 + offset:
                break
            kv_end = min(kv_start + block_kv, skv)
            tiles_visited += 1
            cols = np.arange(kv_start, kv_end)
            if causal:
                visible = cols[None, :] <= rows[:, None] + offset
            else:
                visible = np.ones((rows.size, cols.size), dtype=bool)
            live = visible.any(axis=1)  # rows with at least one visible key
            if not live.any():
                continue
            s = (q[q_start:q_end] @ k[kv_start:kv_end].T) * scale
            s = np.where(visible, s, -math.inf)
            tile_max = s.max(axis=1)
            m_new = np.where(live, np.maximum(m, tile_max), m)
            with np.errstate(invalid="ignore"):
                rescale = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
            # rows without a visible key keep m = -inf; give them a finite
            # shift so that exp(-inf - shift) is a clean 0
            shift = np.where(np.isneginf(m_new), 0.0, m_new)
            p = np.exp(s - shift[:, None])
            p = np.where(visible, p, 0.0)
            acc_scale = rescale if rescale_previous_acc else np.ones_like(rescale)
            a_new = a * acc_scale[:, None] + p @ v[kv_start:kv_end]
            l_new = l * rescale + p.sum(axis=1)
            a = np.where(live[:, None], a_new, a)
            l = np.where(live, l_new, l)
            m = m_new
        nonzero = l > 0
        with np.errstate(divide="ignore", invalid="ignore"):
            out[q_start:q_end] = np.where(nonzero[:, None], a / np.where(nonzero, l, 1.0)[:, None], 0.0)
            lse[q_start:q_end] = np.where(nonzero, m + np.log(np.where(nonzero, l, 1.0)), -math.inf)
    return out, lse, tiles_visited


def tiled_attention(q, k, v, block_q: int = 16, block_kv: int = 16,
                    causal: bool = True, scale: float | None = None,
                    rescale_previous_acc: bool = True):
    """Tiled online-softmax attention over inputs [..., Sq, d] / [..., Skv, d].

    Returns ``(out, lse, meta)``; ``meta`` carries the page's counters:
    ``tiles_visited`` (summed over heads), ``max_sram_score_tile_elements``
    (block_q * block_kv) and ``materialized_nxn_elements`` (always 0).
    ``rescale_previous_acc=False`` reproduces the page's deliberate fault:
    the normaliser is still rescaled but the output accumulator is not."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if block_q < 1 or block_kv < 1:
        raise ValueError("block sizes must be positive")
    lead = q.shape[:-2]
    sq, d = q.shape[-2:]
    skv = k.shape[-2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qf = q.reshape(-1, sq, d)
    kf = k.reshape(-1, skv, d)
    vf = v.reshape(-1, skv, d)
    out = np.zeros_like(qf)
    lse = np.zeros(qf.shape[:2])
    visited = 0
    for h in range(qf.shape[0]):
        o_h, l_h, t_h = _one_head(qf[h], kf[h], vf[h], block_q, block_kv, causal,
                                  scale, rescale_previous_acc)
        out[h], lse[h] = o_h, l_h
        visited += t_h
    meta = {"materialized_nxn_elements": 0,
            "max_sram_score_tile_elements": block_q * block_kv,
            "tiles_visited": visited}
    return out.reshape(lead + (sq, d)), lse.reshape(lead + (sq,)), meta


def block_normalised_average(scores, values, blocks):
    """The deliberately wrong baseline of huhohoo "tiled-online-softmax"
    ("A failing baseline"): softmax each block of scalar scores on its own,
    form that block's weighted value, then give every block equal weight.

    ``scores`` and ``values`` are 1-D; ``blocks`` is a list of index lists."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    outs = []
    for idx in blocks:
        s = scores[list(idx)]
        w = np.exp(s - s.max())
        w = w / w.sum()
        outs.append(float(w @ values[list(idx)]))
    return sum(outs) / len(outs)
