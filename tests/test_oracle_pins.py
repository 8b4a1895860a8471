"""Pins for the fp64 oracle (O1) against facts fixed outside the oracle: values
the pages print, closed forms, library special cases and invariants.

Each test is chosen so that a plausible slip in the oracle (wrong scale, a
transposed operand, an off-by-one causal limit, a missing max shift, a wrong
normaliser or log-sum-exp) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
from scipy import special

import oracle
import qkv_inputs
from conftest import load_golden


# --------------------------------------------------------------------------
# values printed on the pages
# --------------------------------------------------------------------------

def test_p1_printed_sample_rows():
    """aiml.sh "verify-tiled-attention", recorded equivalence_check: the
    first four outputs of row 0 and of the last row, causal, N=64, d=16,
    seed 42, printed to 6 decimals."""
    g = load_golden("p1_equivalence_check.json")
    q, k, v = qkv_inputs.make_qkv(64, 16, 42)
    o, lse = oracle.attention(q, k, v, causal=True)
    assert o.shape == (64, 16)
    assert [round(x, 6) for x in o[0, :4]] == g["sample_row0_first4"]
    assert [round(x, 6) for x in o[-1, :4]] == g["sample_last_row_first4"]
    # the page's row 0 is exactly v[0]: a causal first row sees only key 0
    assert np.array_equal(o[0], np.asarray(v[0]))


@pytest.mark.parametrize("seed", [42, 7])
def test_uniform_generator_is_the_pages_make_qkv(seed):
    """The array generator used for the single-head and decode-like inputs
    draws exactly what aiml.sh "verify-tiled-attention" make_qkv draws: with
    one (batch, head) slice and Sq = Skv it returns the same q, k and v,
    element for element, as the page's list generator (whose seed-42 output
    the printed sample rows pin above)."""
    q_l, k_l, v_l = qkv_inputs.make_qkv(64, 16, seed)
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 64, 64, 16, seed)
    for arr, lists in ((q, q_l), (k, k_l), (v, v_l)):
        assert arr.shape == (1, 1, 64, 16)
        assert np.array_equal(arr[0, 0], np.asarray(lists, dtype=np.float64))


def test_p1_retained_element_count():
    """The page's dense reference keeps 4160 score+probability elements for
    causal N=64, i.e. 2080 visible (query, key) pairs.  With q = 0 every
    visible score is 0, so lse_i = ln(#visible keys of row i) and the sum of
    exp(lse) counts the visible pairs."""
    g = load_golden("p1_equivalence_check.json")
    q = np.zeros((64, 16))
    k = np.asarray(qkv_inputs.make_qkv(64, 16, 42)[1])
    v = np.asarray(qkv_inputs.make_qkv(64, 16, 42)[2])
    _, lse = oracle.attention(q, k, v, causal=True)
    assert round(float(np.exp(lse).sum())) * 2 == g["standard_materialized_elements"]


# --------------------------------------------------------------------------
# the worked example of huhohoo "tiled-online-softmax"
# --------------------------------------------------------------------------

def _worked_example_inputs():
    g = load_golden("p3_worked_example.json")
    # one query with q = [1] and scale 1 feeds the scalar scores directly
    q = np.array([[1.0]])
    k = np.array(g["scores"], dtype=np.float64).reshape(-1, 1)
    v = np.array(g["values"], dtype=np.float64).reshape(-1, 1)
    return g, q, k, v


def test_worked_example_full_softmax_closed_form():
    g, q, k, v = _worked_example_inputs()
    o, lse = oracle.attention(q, k, v, causal=False, scale=1.0)
    # closed form, rearranged: 5 - (4 e^-20 + 2 e^-10) / (1 + e^-10 + e^-20)
    e10, e20 = math.exp(-10.0), math.exp(-20.0)
    full = 5.0 - (4.0 * e20 + 2.0 * e10) / (1.0 + e10 + e20)
    assert abs(o[0, 0] - full) <= 1e-15 * full
    assert abs(o[0, 0] - 4.9999091960185416) <= 1e-15 * full
    lse_closed = 20.0 + math.log1p(e10 + e20)
    assert abs(lse[0] - lse_closed) <= 1e-15 * lse_closed
    assert abs(lse[0] - 20.000045400960278) <= 1e-15 * lse_closed


def test_worked_example_wrong_baseline_differs():
    g, q, k, v = _worked_example_inputs()
    wrong = oracle.block_normalised_average(g["scores"], g["values"],
                                            g["wrong_baseline_blocks"])
    # closed form of the equal-weight average: 4 - 1 / (1 + e^10)
    assert abs(wrong - (4.0 - 1.0 / (1.0 + math.exp(10.0)))) <= 1e-15
    o, _ = oracle.attention(q, k, v, causal=False, scale=1.0)
    assert abs(o[0, 0] - wrong) > 0.99


# --------------------------------------------------------------------------
# library special cases (torch / scipy softmax and logsumexp in fp64)
# --------------------------------------------------------------------------

def _torch_reference(q, k, v, causal, scale):
    q, k, v = (torch.as_tensor(np.asarray(x), dtype=torch.float64) for x in (q, k, v))
    s = (q @ k.transpose(-2, -1)) * scale
    if causal:
        sq, skv = s.shape[-2], s.shape[-1]
        i = torch.arange(sq)[:, None]
        j = torch.arange(skv)[None, :]
        s = s.masked_fill(j > i + (skv - sq), float("-inf"))
    return (torch.softmax(s, dim=-1) @ v).numpy(), torch.logsumexp(s, dim=-1).numpy()


CASES = [
    # (name, generator, causal)
    ("c1-causal", lambda: qkv_inputs.uniform_qkv(1, 1, 64, 64, 32, 42), True),
    ("c1-full", lambda: qkv_inputs.uniform_qkv(1, 1, 64, 64, 32, 42), False),
    ("c2-1024", lambda: qkv_inputs.uniform_qkv(1, 1, 8, 1024, 32, 1), False),
    ("c3", lambda: tuple(t.numpy() for t in qkv_inputs.normal_qkv(2, 4, 512, 512, 64, 0)), False),
    ("ragged-causal", lambda: qkv_inputs.uniform_qkv(2, 3, 37, 53, 16, 5), True),
    ("sq>skv-causal", lambda: qkv_inputs.uniform_qkv(1, 2, 40, 24, 8, 6), True),
]


@pytest.mark.parametrize("name,gen,causal", CASES, ids=[c[0] for c in CASES])
def test_matches_torch_softmax_fp64(name, gen, causal):
    q, k, v = gen()
    scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = oracle.attention(q, k, v, causal=causal)
    o_ref, lse_ref = _torch_reference(q, k, v, causal, scale)
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), finite)
    assert np.allclose(o[finite], o_ref[finite], rtol=0, atol=1e-12)
    assert np.allclose(lse[finite], lse_ref[finite], rtol=0, atol=1e-12)
    # rows without any visible key (torch gives NaN there): zero output and
    # -inf lse, the reading chosen for such rows
    assert np.all(o[~finite] == 0.0)
    assert np.all(lse[~finite] == -math.inf)


def test_matches_scipy_softmax_fp64():
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 8, 256, 32, 2)
    q, k, v = q[0, 0], k[0, 0], v[0, 0]
    s = (q @ k.T) / math.sqrt(32)
    o_ref = special.softmax(s, axis=-1) @ v
    lse_ref = special.logsumexp(s, axis=-1)
    o, lse = oracle.attention(q, k, v)
    assert np.max(np.abs(o - o_ref)) <= 1e-13
    assert np.max(np.abs(lse - lse_ref)) <= 1e-13


# --------------------------------------------------------------------------
# closed forms on tiny inputs
# --------------------------------------------------------------------------

def test_single_key_returns_its_value():
    rng = np.random.default_rng(3)
    q, k, v = rng.normal(size=(5, 3)), rng.normal(size=(1, 3)), rng.normal(size=(1, 3))
    o, lse = oracle.attention(q, k, v, scale=0.7)
    assert np.array_equal(o, np.repeat(v, 5, axis=0))
    assert np.allclose(lse, 0.7 * (q @ k[0]), rtol=0, atol=1e-15)


def test_two_keys_sigmoid_form():
    """With two keys, o = v0 + (v1 - v0) * sigmoid(s1 - s0) and
    lse = max(s) + log1p(exp(-|s1 - s0|))."""
    rng = np.random.default_rng(4)
    q, k, v = rng.normal(size=(3, 2)), rng.normal(size=(2, 2)), rng.normal(size=(2, 2))
    scale = 0.9
    o, lse = oracle.attention(q, k, v, scale=scale)
    for i in range(3):
        s0, s1 = scale * (q[i] @ k[0]), scale * (q[i] @ k[1])
        w = special.expit(s1 - s0)
        assert np.allclose(o[i], v[0] + (v[1] - v[0]) * w, rtol=0, atol=1e-15)
        assert abs(lse[i] - (max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0))))) <= 1e-15


def test_causal_two_by_two():
    """Causal 2x2: row 0 sees key 0 only, row 1 both keys."""
    rng = np.random.default_rng(5)
    q, k, v = rng.normal(size=(2, 2)), rng.normal(size=(2, 2)), rng.normal(size=(2, 2))
    o, lse = oracle.attention(q, k, v, causal=True, scale=1.0)
    assert np.array_equal(o[0], v[0])
    assert lse[0] == q[0] @ k[0]
    w = special.expit(q[1] @ k[1] - q[1] @ k[0])
    assert np.allclose(o[1], v[0] + (v[1] - v[0]) * w, rtol=0, atol=1e-15)


def test_p1_overflow_case():
    """aiml.sh "verify-tiled-attention", test_naive_softmax_overflows_without
    _max_shift: logits of 500-valued queries overflow exp() without the max
    shift; with it the result is finite and equals the two-key closed form."""
    q = [[500.0, 500.0], [500.0, 500.0]]
    k = [[1.0, 1.0], [2.0, 2.0]]
    v = [[1.0, 0.0], [0.0, 1.0]]
    o_bad, _ = oracle.attention(q, k, v, causal=False, subtract_max=False)
    assert not np.all(np.isfinite(o_bad))
    o, lse = oracle.attention(q, k, v, causal=False)
    delta = 1000.0 / math.sqrt(2.0)  # s1 - s0 with scale 1/sqrt(2)
    expect = np.array([special.expit(-delta), special.expit(delta)])
    assert np.all(np.isfinite(o))
    assert np.allclose(o, np.vstack([expect, expect]), rtol=1e-15, atol=0)
    assert np.allclose(lse, 2000.0 / math.sqrt(2.0), rtol=1e-15, atol=0)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_identity_values_give_probability_rows(causal):
    """V = I (Skv = d) makes O equal to the probability matrix: rows sum to 1,
    entries are non-negative and masked entries are exactly 0."""
    d = 24
    q, k, _ = qkv_inputs.uniform_qkv(1, 1, d, d, d, 11)
    o, _ = oracle.attention(q[0, 0], k[0, 0], np.eye(d), causal=causal)
    assert np.all(np.abs(o.sum(axis=1) - 1.0) <= 1e-14)
    assert np.all(o >= 0.0)
    if causal:
        assert np.all(np.triu(o, 1) == 0.0)


def test_constant_values_give_constant_output():
    q, k, _ = qkv_inputs.uniform_qkv(1, 2, 33, 33, 8, 12)
    v = np.broadcast_to(np.arange(8.0) - 3.5, k.shape).copy()
    o, _ = oracle.attention(q, k, v, causal=True)
    assert np.max(np.abs(o - v[..., :1, :])) <= 1e-14


def test_shift_invariance():
    """Adding c_i to every score of query row i leaves the output unchanged
    and shifts lse by c_i.  The shift is built by appending one feature:
    q' = [q, c_i / scale], k' = [k, 1]."""
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 20, 30, 8, 13)
    q, k, v = q[0, 0], k[0, 0], v[0, 0]
    scale = 0.5
    c = np.linspace(-40.0, 40.0, 20)
    q2 = np.hstack([q, (c / scale)[:, None]])
    k2 = np.hstack([k, np.ones((30, 1))])
    v2 = np.hstack([v, np.zeros((30, 1))])  # one head width for q, k and v
    o1, l1 = oracle.attention(q, k, v, scale=scale)
    o2, l2 = oracle.attention(q2, k2, v2, scale=scale)
    assert np.all(o2[:, 8] == 0.0)
    assert np.max(np.abs(o1 - o2[:, :8])) <= 1e-13
    assert np.max(np.abs((l2 - l1) - c)) <= 1e-12


def test_key_permutation_invariance():
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 16, 40, 8, 14)
    perm = np.random.default_rng(0).permutation(40)
    o1, l1 = oracle.attention(q, k, v)
    o2, l2 = oracle.attention(q, k[..., perm, :], v[..., perm, :])
    assert np.max(np.abs(o1 - o2)) <= 1e-14
    assert np.max(np.abs(l1 - l2)) <= 1e-14


def test_scale_multiplies_scores():
    q, k, v = qkv_inputs.uniform_qkv(1, 1, 12, 12, 8, 15)
    o1, l1 = oracle.attention(q, k, v, causal=True, scale=0.25)
    o2, l2 = oracle.attention(q * 0.25, k, v, causal=True, scale=1.0)
    assert np.max(np.abs(o1 - o2)) <= 1e-14
    assert np.max(np.abs(l1 - l2)) <= 1e-14


@pytest.mark.parametrize("sq,skv", [(7, 7), (5, 9), (9, 5), (1, 6)])
def test_zero_queries_average_visible_values(sq, skv):
    """q = 0 gives equal weights: o_i is the mean of the visible values and
    lse_i = ln(#visible).  This pins the causal visibility rule: key j is
    visible to query i iff j <= i + (Skv - Sq); rows with no visible key
    return 0 and -inf."""
    rng = np.random.default_rng(sq * 100 + skv)
    q = np.zeros((sq, 4))
    k = rng.normal(size=(skv, 4))
    v = rng.normal(size=(skv, 4))
    o, lse = oracle.attention(q, k, v, causal=True)
    for i in range(sq):
        n = min(skv, max(0, i + 1 + skv - sq))
        if n == 0:
            assert np.all(o[i] == 0.0) and lse[i] == -math.inf
        else:
            assert np.allclose(o[i], v[:n].mean(axis=0), rtol=0, atol=1e-15)
            assert abs(lse[i] - math.log(n)) <= 1e-15


def test_thread_count_does_not_change_bits():
    q, k, v = qkv_inputs.uniform_qkv(2, 2, 50, 50, 16, 16)
    o1, l1 = oracle.attention(q, k, v, causal=True, nthreads=1)
    o8, l8 = oracle.attention(q, k, v, causal=True, nthreads=8)
    assert np.array_equal(o1, o8) and np.array_equal(l1, l8)


def test_rows_entry_matches_full_entry():
    q, k, v = qkv_inputs.uniform_qkv(2, 3, 40, 56, 16, 17)
    o, lse = oracle.attention(q, k, v, causal=True)
    rows = [(0, 0), (5, 39), (3, 17), (1, 1)]
    o_r, l_r = oracle.attention_rows(q, k, v, rows, causal=True)
    of, lf = o.reshape(6, 40, 16), lse.reshape(6, 40)
    for n, (bh, i) in enumerate(rows):
        assert np.array_equal(o_r[n], of[bh, i])
        assert l_r[n] == lf[bh, i]


def test_access_model_matches_printed_sweep():
    """aiml.sh "verify-tiled-attention", recorded hbm_traffic_sweep."""
    g = load_golden("p1_hbm_traffic_sweep.json")
    for row in g["rows"]:
        r = oracle.estimate_hbm_bytes(row["seq_len"], num_heads=32, head_dim=128,
                                      bytes_per_elem=2)
        assert r["qkvo_compulsory_bytes_mb"] == row["standard_qkv_o_mb"]
        assert r["standard_nxn_matrix_hbm_mb"] == row["standard_nxn_matrix_hbm_mb"]
        assert r["standard_total_hbm_mb"] == row["standard_total_hbm_mb"]
        assert r["tiled_logical_access_mb_no_cache_reuse"] == \
            row["tiled_logical_access_mb_no_cache_reuse"]
        assert r["num_q_blocks"] == row["num_q_blocks"]


def test_access_model_page_properties():
    """aiml.sh "verify-tiled-attention", test_access_count_includes_repeated
    _kv_reads: tiled logical bytes exceed the compulsory bytes, and grow more
    than 8x from 4k to 32k tokens."""
    small = oracle.estimate_hbm_bytes(4096)
    large = oracle.estimate_hbm_bytes(32768)
    assert small["tiled_logical_access_mb_no_cache_reuse"] > small["qkvo_compulsory_bytes_mb"]
    assert (large["tiled_logical_access_mb_no_cache_reuse"]
            / small["tiled_logical_access_mb_no_cache_reuse"]) > 8
