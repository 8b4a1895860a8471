"""Pins for the oracle's merge of partial results (``oracle.merge_partials``).

The merge is pinned to the plain attention definition (O1 over all keys must
equal the merge of O1 over any partition of the keys), to closed forms of the
worked example of huhohoo "tiled-online-softmax" ("A failing baseline"), and
to the empty-part and ordering properties.  A dropped rescale factor, a wrong
sign in an exponent, a swapped weight or a missing normalisation fails the
partition test.
"""
import math

import numpy as np
import pytest

import oracle
import qkv_inputs
from conftest import load_golden


def _parts(q, k, v, bounds, scale=None):
    """O1 over each key range of `bounds`: (o_parts, lse_parts), rows flattened."""
    os_, ls_ = [], []
    for a, b in bounds:
        o, lse = oracle.attention(q, k[..., a:b, :], v[..., a:b, :], scale=scale)
        os_.append(o.reshape(-1, o.shape[-1]))
        ls_.append(lse.reshape(-1))
    return np.stack(os_), np.stack(ls_)


@pytest.mark.parametrize("bounds", [
    [(0, 64), (64, 128)],
    [(0, 7), (7, 70), (70, 128)],
    [(0, 1), (1, 2), (2, 128)],
    [(100, 128), (0, 100)],          # order of the parts is free
])
def test_merge_of_key_partition_equals_full_attention(bounds):
    q, k, v = (np.asarray(x) for x in qkv_inputs.normal_qkv(2, 3, 9, 128, 32, seed=5))
    o_ref, lse_ref = oracle.attention(q, k, v)
    o_p, l_p = _parts(q, k, v, bounds)
    o, lse = oracle.merge_partials(o_p, l_p)
    assert np.abs(o - o_ref.reshape(-1, 32)).max() <= 1e-13
    assert np.abs(lse - lse_ref.reshape(-1)).max() <= 1e-13


def test_merge_large_score_gap_keeps_precision():
    """Scores 50x larger (the decode stress variant): the shift by the running
    maximum keeps every exponential finite."""
    q, k, v = (np.asarray(x) for x in qkv_inputs.uniform_qkv(1, 1, 8, 256, 32, 1))
    q = q * 50.0
    o_ref, lse_ref = oracle.attention(q, k, v)
    o_p, l_p = _parts(q, k, v, [(0, 100), (100, 101), (101, 256)])
    o, lse = oracle.merge_partials(o_p, l_p)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(o - o_ref.reshape(-1, 32)).max() <= 1e-12
    assert np.abs(lse - lse_ref.reshape(-1)).max() <= 1e-12


def test_worked_example_block_merge():
    """Scores 0, 10 in one block and 20 in the other, values 1, 3, 5.  The
    merge reaches the full softmax, (e^-20 + 3 e^-10 + 5) / (1 + e^-10 + e^-20),
    and lse = 20 + ln(1 + e^-10 + e^-20); the page's averaged baseline differs
    by about 1."""
    g = load_golden("p3_worked_example.json")
    s, val = g["scores"], g["values"]
    lse_a = math.log(math.exp(s[0]) + math.exp(s[1]))
    o_a = (val[0] * math.exp(s[0]) + val[1] * math.exp(s[1])) / (math.exp(s[0]) + math.exp(s[1]))
    o_p = np.array([[[o_a]], [[val[2]]]])
    l_p = np.array([[lse_a], [s[2]]])
    o, lse = oracle.merge_partials(o_p, l_p)
    full = (math.exp(-20) + 3 * math.exp(-10) + 5) / (1 + math.exp(-10) + math.exp(-20))
    assert abs(o[0, 0] - full) <= 1e-15
    assert abs(lse[0] - (20 + math.log1p(math.exp(-10) + math.exp(-20)))) <= 1e-14
    wrong = (o_a + val[2]) / 2  # normalise each block, then average
    assert abs(o[0, 0] - wrong) > 0.99


def test_single_part_is_identity_and_empty_parts_vanish():
    rng = np.random.default_rng(3)
    o1 = rng.standard_normal((1, 5, 4))
    l1 = rng.standard_normal((1, 5))
    o, lse = oracle.merge_partials(o1, l1)
    assert np.array_equal(o, o1[0]) and np.allclose(lse, l1[0], rtol=0, atol=1e-15)
    # an extra part with lse = -inf (no visible key) changes nothing
    o2 = np.concatenate([o1, rng.standard_normal((1, 5, 4))])
    l2 = np.concatenate([l1, np.full((1, 5), -math.inf)])
    o, lse = oracle.merge_partials(o2, l2)
    assert np.allclose(o, o1[0], rtol=0, atol=1e-15) and np.allclose(lse, l1[0], rtol=0, atol=1e-15)
    # every part empty: output 0, lse -inf
    o, lse = oracle.merge_partials(np.ones((3, 2, 4)), np.full((3, 2), -math.inf))
    assert np.array_equal(o, np.zeros((2, 4))) and np.all(lse == -math.inf)


def test_equal_parts_average_with_log_two():
    """Two parts with the same lse weigh equally: the merge is their mean and
    lse grows by ln 2."""
    o_p = np.array([[[1.0, -2.0]], [[3.0, 4.0]]])
    l_p = np.array([[0.25], [0.25]])
    o, lse = oracle.merge_partials(o_p, l_p)
    assert np.allclose(o, [[2.0, 1.0]], rtol=0, atol=1e-15)
    assert abs(lse[0] - (0.25 + math.log(2.0))) <= 1e-15
