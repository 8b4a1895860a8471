"""The tiled online-softmax algorithm (O2) against the pinned oracle (O1).

These restate the checks the pages run on their CPU implementations: the
tile-size sweep and the two failure boundaries of aiml.sh
"verify-tiled-attention" (test_lab.py), the block-size-7 and large-score
exercises of huhohoo "tiled-online-softmax", and its recorded comparison
(three seeds, 64/256/1024 keys, eight query rows, width 32, block 32).
"""
import math

import numpy as np
import pytest

import oracle
import qkv_inputs
from conftest import load_golden


def test_p1_tiles_visited_and_equivalence():
    g = load_golden("p1_equivalence_check.json")
    q, k, v = qkv_inputs.make_qkv(64, 16, 42)
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    o, _, meta = oracle.tiled_attention(q, k, v, 16, 16, causal=True)
    assert meta["tiles_visited"] == g["flash_tiles_visited"]
    assert meta["max_sram_score_tile_elements"] == g["flash_sram_tile_elements"]
    assert meta["materialized_nxn_elements"] == 0
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert [round(x, 6) for x in o[0, :4]] == g["sample_row0_first4"]
    assert [round(x, 6) for x in o[-1, :4]] == g["sample_last_row_first4"]


@pytest.mark.parametrize("bq,bkv", [(8, 8), (16, 16), (13, 19), (32, 8), (7, 7),
                                    (1, 1), (64, 64), (5, 64)])
def test_p1_tile_sweep(bq, bkv):
    """test_tiled_flash_attention_matches_standard_attention_across_tile_sizes
    (seed 7, N=64, d=16, causal) plus block 7 and the degenerate sizes."""
    q, k, v = qkv_inputs.make_qkv(64, 16, 7)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    o, lse, meta = oracle.tiled_attention(q, k, v, bq, bkv, causal=True)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12
    assert meta["materialized_nxn_elements"] == 0


def test_p1_overflow_case_tiled():
    q = [[500.0, 500.0], [500.0, 500.0]]
    k = [[1.0, 1.0], [2.0, 2.0]]
    v = [[1.0, 0.0], [0.0, 1.0]]
    o_ref, _ = oracle.attention(q, k, v, causal=False)
    o, _, _ = oracle.tiled_attention(q, k, v, 1, 1, causal=False)
    assert np.max(np.abs(o - o_ref)) < 1e-12


def test_p1_forgetting_rescale_corrupts_output():
    """test_forgetting_output_rescaling_across_tiles_corrupts_attention:
    seed 99, N=32, d=8, the last key set to 4.0 so the running max rises on a
    later tile; blocks of 8.  Correct < 1e-12, without the rescale > 0.1."""
    q, k, v = qkv_inputs.make_qkv(32, 8, 99)
    k[-1] = [4.0] * 8
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    good, _, _ = oracle.tiled_attention(q, k, v, 8, 8, causal=True)
    bad, _, _ = oracle.tiled_attention(q, k, v, 8, 8, causal=True,
                                       rescale_previous_acc=False)
    assert np.max(np.abs(o_ref - good)) < 1e-12
    assert np.max(np.abs(o_ref - bad)) > 0.1


def test_worked_example_tiled_blocks():
    """The scores 0/10/20 split into blocks {0, 10} and {20}: the online
    merge recovers the full softmax; the equal-weight average does not."""
    g = load_golden("p3_worked_example.json")
    q = np.array([[1.0]])
    k = np.array(g["scores"]).reshape(-1, 1)
    v = np.array(g["values"]).reshape(-1, 1)
    o_ref, lse_ref = oracle.attention(q, k, v, scale=1.0)
    o, lse, meta = oracle.tiled_attention(q, k, v, 1, 2, causal=False, scale=1.0)
    assert meta["tiles_visited"] == 2
    assert abs(o[0, 0] - o_ref[0, 0]) <= 1e-15
    assert abs(lse[0] - lse_ref[0]) <= 1e-14
    bad, _, _ = oracle.tiled_attention(q, k, v, 1, 2, causal=False, scale=1.0,
                                       rescale_previous_acc=False)
    assert abs(bad[0, 0] - o_ref[0, 0]) > 0.1


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("skv", [64, 256, 1024])
def test_p3_recorded_comparison(seed, skv):
    """Eight query rows, width 32, block 32, no mask; the page records a
    maximum dense/tiled discrepancy of 3.33e-16 over its nine groups."""
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 8, skv, 32, seed)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False)
    o, lse, _ = oracle.tiled_attention(q, k, v, 32, 32, causal=False)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12
    # the large-score exercise: scores scaled by 50 stay finite and agree
    o50_ref, _ = oracle.attention(q * 50.0, k, v, causal=False)
    o50, _, _ = oracle.tiled_attention(q * 50.0, k, v, 32, 32, causal=False)
    assert np.all(np.isfinite(o50))
    assert np.max(np.abs(o50 - o50_ref)) < 1e-12


@pytest.mark.parametrize("sq,skv", [(37, 53), (53, 37), (1, 9), (9, 1), (64, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_and_rectangular(sq, skv, causal):
    q, k, v = qkv_inputs.uniform_qkv(1, 2, sq, skv, 8, sq + skv)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    for bq, bkv in ((7, 7), (16, 5), (64, 64)):
        o, lse, _ = oracle.tiled_attention(q, k, v, bq, bkv, causal=causal)
        assert np.max(np.abs(o - o_ref)) < 1e-12
        finite = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), finite)
        assert np.max(np.abs(lse[finite] - lse_ref[finite]), initial=0.0) < 1e-12


def test_config1_tiles_and_missing_rescale():
    """Single head, N=64, d=32, seed 42, tiles 16x16 and 7x7: both agree with
    the oracle; dropping the accumulator rescale is caught."""
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 64, 64, 32, 42)
    for causal in (False, True):
        o_ref, _ = oracle.attention(q, k, v, causal=causal)
        for b in (16, 7):
            o, _, _ = oracle.tiled_attention(q, k, v, b, b, causal=causal)
            assert np.max(np.abs(o - o_ref)) < 1e-12
    # a late large key makes the running maximum rise on a later tile
    k2 = k.copy()
    k2[0, 0, -1, :] = 4.0
    o_ref, _ = oracle.attention(q, k2, v, causal=False)
    bad, _, _ = oracle.tiled_attention(q, k2, v, 16, 16, causal=False,
                                       rescale_previous_acc=False)
    assert np.max(np.abs(o_ref - bad)) > 0.1
