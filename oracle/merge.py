"""Merge of partial attention results over disjoint key sets -- TEST
INFRASTRUCTURE ONLY (see the package docstring).

A partial result of one query row over a subset of the keys is the pair
(o_part, lse_part): the softmax-weighted average of the subset's values and
the log-sum-exp of the subset's scaled scores.  It is the running state
(m, l, a) of the online softmax written as m = lse_part, l = 1,
a = o_part, since exp(lse_part) = l * exp(m) for the subset's own max m.

Combining states is the update of huhohoo "tiled-online-softmax" ("Online
normalization") applied to whole states instead of single tiles, the same
step aiml.sh "verify-tiled-attention" (tiled_flash_attention) takes when a
new key block raises the running maximum:

    m_new = max(m, m_part)
    a     = a * exp(m - m_new) + a_part * exp(m_part - m_new)
    l     = l * exp(m - m_new) + l_part * exp(m_part - m_new)
    out   = a / l,  lse = m_new + ln l

A part with lse = -inf (no visible key) contributes nothing; a row where
every part is -inf gets out = 0 and lse = -inf, like a row with no visible
key.  Everything is fp64 and parts are folded in the order given.
"""
from __future__ import annotations

import math

import numpy as np


def merge_partials(o_parts, lse_parts):
    """o_parts [n_parts, rows, d], lse_parts [n_parts, rows] (natural log)
    -> (o [rows, d], lse [rows]) in fp64."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    if o_parts.ndim != 3 or lse_parts.shape != o_parts.shape[:2]:
        raise ValueError("shapes: o_parts %s lse_parts %s" % (o_parts.shape, lse_parts.shape))
    n, rows, d = o_parts.shape
    m = np.full((rows,), -math.inf)
    l = np.zeros((rows,))
    a = np.zeros((rows, d))
    for p in range(n):
        m_part = lse_parts[p]
        m_new = np.maximum(m, m_part)
        live = m_new > -math.inf  # rows that have seen at least one key
        r_old = np.zeros((rows,))
        r_part = np.zeros((rows,))
        r_old[live] = np.exp(m[live] - m_new[live])      # exp(-inf) = 0 for empty states
        r_part[live] = np.exp(m_part[live] - m_new[live])
        a = a * r_old[:, None] + o_parts[p] * r_part[:, None]
        l = l * r_old + r_part
        m = m_new
    out = np.zeros((rows, d))
    lse = np.full((rows,), -math.inf)
    seen = l > 0
    out[seen] = a[seen] / l[seen][:, None]
    lse[seen] = m[seen] + np.log(l[seen])
    return out, lse
