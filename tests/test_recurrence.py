"""Pins of the oracle's scalar model of the online-softmax recurrence.

The model follows the block-wise algorithm of "tm_flash_attention_math",
section "The block-wise update, and the full algorithm".  It is checked
against the pages' two worked examples, the stability and exactness claims
(section "Proof of numerical stability", "Proof of exactness"), and the
three-pass fp64 oracle; each of the four pitfalls the page lists is planted in
the model and must be caught.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.recurrence import PITFALLS, blocks_of, online_softmax_attention


def _three_pass(scores, values, visible=None):
    """The fp64 oracle on one query.  With one-hot keys (K = I, d = n) the score
    of key j is q[j], so the raw scores go in as q.  A masked key carries no
    probability mass, so masked keys are dropped before the call (the oracle
    itself knows only the causal mask)."""
    if visible is not None:
        keep = [j for j in range(len(scores)) if visible[j]]
        scores = [scores[j] for j in keep]
        values = [values[j] for j in keep]
    s = np.asarray(scores, dtype=np.float64)
    n = len(s)
    vals = np.asarray(values, dtype=np.float64).reshape(n, -1)
    dv = vals.shape[1]
    d = max(n, dv)
    Q = np.zeros((1, 1, n, d))
    Q[0, 0, :, :n] = s  # every row asks the same question; row 0 is read
    K = np.zeros((1, 1, n, d))
    K[0, 0, :, :n] = np.eye(n)
    V = np.zeros((1, 1, n, d))
    V[0, 0, :, :dv] = vals
    o, lse = oracle.attention_fwd(Q, K, V, 1.0, False)
    return o[0, 0, 0, :dv], lse[0, 0, 0]


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_four_key_example_block_by_block(golden_dir):
    g = _load(golden_dir, "four_key_example.json")
    tol = g["per_block_tol"]
    o, m, l, trace = online_softmax_attention(g["scores"], [[x] for x in g["values"]], g["blocks"])
    for got, want in zip(trace, g["per_block"]):
        assert got["m_blk"] == want["m_blk"] and got["m_new"] == want["m_new"]
        assert abs(got["alpha"] - want["alpha"]) <= tol["alpha"]
        np.testing.assert_allclose(got["p"], want["p"], atol=tol["p"])
        assert abs(got["l"] - want["l"]) <= tol["l"]
        assert abs(got["o_tilde"][0] - want["o_tilde"]) <= tol["o_tilde"]
    assert abs(l - g["l"]["value"]) <= g["l"]["tol"]
    assert abs(o[0] - g["o"]["value"]) <= g["o"]["tol"]


def test_eight_score_example_running_state(golden_dir):
    g = _load(golden_dir, "eight_score_example.json")
    scores = g["blocks"][0] + g["blocks"][1]
    _, _, _, trace = online_softmax_attention(scores, [[0.0]] * 8, blocks_of(8, 4))
    for t, m_exp, l_exp in zip(trace, g["running_max"], g["running_sum"]):
        assert t["m_new"] == m_exp
        assert abs(t["l"] - l_exp) <= g["tol_sum"]


def _random_case(seed, n=23, dv=3, spread=6.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n) * spread).tolist(), rng.standard_normal((n, dv)).tolist()


@pytest.mark.parametrize("size", [1, 2, 3, 5, 8, 23, 64])
def test_exact_for_any_block_size(size):
    scores, values = _random_case(100 + size)
    o_ref, lse_ref = _three_pass(scores, values)
    o, m, l, _ = online_softmax_attention(scores, values, blocks_of(len(scores), size))
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-14)
    assert abs(m + math.log(l) - lse_ref) < 1e-13


@pytest.mark.parametrize("seed", range(5))
def test_exact_for_any_block_order(seed):
    scores, values = _random_case(200 + seed)
    rng = np.random.default_rng(seed)
    nb = len(blocks_of(len(scores), 4))
    o_ref, lse_ref = _three_pass(scores, values)
    o, m, l, _ = online_softmax_attention(scores, values, blocks_of(len(scores), 4, rng.permutation(nb)))
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-14)
    assert abs(m + math.log(l) - lse_ref) < 1e-13


def test_every_exp_argument_is_nonpositive_and_alpha_in_unit_interval():
    scores, values = _random_case(300, n=200, spread=40.0)  # far beyond exp's fp32 range
    o, m, l, trace = online_softmax_attention(scores, values, blocks_of(200, 7))
    seen = []
    for i, t in enumerate(trace):
        assert all(a <= 0.0 for a in t["exp_args"])
        assert all(0.0 <= p <= 1.0 for p in t["p"])
        assert (t["alpha"] == 0.0) if i == 0 else (0.0 < t["alpha"] <= 1.0)
        seen += scores[7 * i: 7 * i + 7]
        assert t["m_new"] == max(seen)  # m is the maximum of the scores seen
    assert all(math.isfinite(x) for x in o)


def test_masked_keys_carry_no_mass():
    scores, values = _random_case(400, n=16)
    visible = [j % 3 != 1 for j in range(16)]
    o_ref, lse_ref = _three_pass(scores, values, visible)
    o, m, l, _ = online_softmax_attention(scores, values, blocks_of(16, 4), visible=visible)
    np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-14)
    assert abs(m + math.log(l) - lse_ref) < 1e-13


# ---------------------------------------------------------------- planted pitfalls

PITFALL_CASES = {
    # the maximum rises in the second block, so alpha < 1 matters for o~
    "rescale_l_only": dict(scores=[1.0, 3.0, 2.0, 5.0], visible=None, size=2),
    # a finite start of 0 above every score: exp(s - 0) underflows to 0 in fp64
    "finite_m_init": dict(scores=[-800.0, -790.0, -805.0, -795.0], visible=None, size=2),
    # a masked key far above the visible ones becomes the reference; the
    # visible terms underflow
    "mask_after_max": dict(scores=[0.5, 900.0, -0.25, 1.0], visible=[True, False, True, True], size=4),
    "normalize_per_block": dict(scores=[1.0, 3.0, 2.0, 5.0], visible=None, size=2),
}


@pytest.mark.parametrize("pitfall", PITFALLS)
def test_each_pitfall_is_caught(pitfall):
    case = PITFALL_CASES[pitfall]
    values = [[10.0, -1.0], [20.0, 2.0], [30.0, 0.5], [40.0, -3.0]]
    o_ref, _ = _three_pass(case["scores"], values, case["visible"])
    blocks = blocks_of(4, case["size"])
    good, _, _, _ = online_softmax_attention(case["scores"], values, blocks, case["visible"])
    np.testing.assert_allclose(good, o_ref, rtol=1e-13)
    bad, _, _, _ = online_softmax_attention(case["scores"], values, blocks, case["visible"], pitfall)
    assert not np.allclose(bad, o_ref, rtol=1e-6, atol=1e-6, equal_nan=False), pitfall


# ---------------------------------------------------------------- lazily moved reference

@pytest.mark.parametrize("slack", [0.5, 2.0, 8 * math.log(2.0), 40.0])
@pytest.mark.parametrize("size", [1, 4, 7, 200])
def test_lazily_moved_reference_is_exact_and_bounded(slack, size):
    """Keeping the old reference while the block max rises by at most ``slack``
    gives the three-pass result (any reference works), and no exp argument
    exceeds ``slack``.  The forward kernel uses slack = 8 ln 2 (2^8 in base 2)."""
    scores, values = _random_case(500 + size, n=200, spread=12.0)
    o_ref, lse_ref = _three_pass(scores, values)
    o, m, l, trace = online_softmax_attention(scores, values, blocks_of(200, size), slack=slack)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    assert abs(m + math.log(l) - lse_ref) < 1e-12
    assert max(a for t in trace for a in t["exp_args"]) <= slack + 1e-12
    assert all(0.0 < t["alpha"] <= 1.0 for t in trace[1:])
    # the reference is never below the first block's max, never above the running max
    seen = []
    for i, t in enumerate(trace):
        seen += scores[size * i: size * i + size]
        assert t["m_new"] <= max(seen)
        assert max(seen) - t["m_new"] <= slack


def test_lazy_reference_skips_rescales():
    scores, values = _random_case(600, n=512, spread=1.0)
    _, _, _, exact = online_softmax_attention(scores, values, blocks_of(512, 16))
    _, _, _, lazy = online_softmax_attention(scores, values, blocks_of(512, 16), slack=8 * math.log(2))
    moves = lambda tr: sum(1 for t in tr[1:] if t["alpha"] != 1.0)
    assert moves(lazy) < moves(exact)
    assert moves(lazy) == 0  # N(0,1) scores never climb 5.5 above the first block's max


# ---------------------------------------------------------------- the row softmax oracle

@pytest.mark.parametrize("size", [1, 3, 16, 200])
def test_row_softmax_is_the_recurrence_with_one_hot_values(size):
    """With one-hot value vectors (V = I) the recurrence's output is the softmax
    itself: the row-softmax oracle agrees with the block-wise model for any
    block size, and its LSE with m + ln l."""
    rng = np.random.default_rng(700 + size)
    x = rng.standard_normal(200) * 9.0
    o, m, l, _ = online_softmax_attention(x.tolist(), np.eye(200).tolist(), blocks_of(200, size))
    y, lse = oracle.softmax_rows(x[None])
    np.testing.assert_allclose(y[0], o, rtol=1e-12, atol=1e-15)
    assert abs(lse[0] - (m + math.log(l))) < 1e-12


def test_row_softmax_invariants():
    rng = np.random.default_rng(701)
    x = rng.standard_normal((5, 33)) * 20.0
    y, lse = oracle.softmax_rows(x)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-14)
    y2, lse2 = oracle.softmax_rows(x + 1234.5)               # shift invariance
    np.testing.assert_allclose(y2, y, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(lse2, lse + 1234.5, rtol=1e-14)
    np.testing.assert_allclose(y, np.exp(x - lse[:, None]), rtol=1e-12, atol=1e-300)
    z = np.full((1, 4), -np.inf)
    yz, lz = oracle.softmax_rows(z)                          # nothing visible
    assert np.all(yz == 0.0) and lz[0] == -np.inf
