"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Nothing here compares the oracle with a retyped copy of its own formula:
each check is a printed worked example, a closed form, an invariant, an
independent library routine (torch's fp64 CPU attention and autograd), or
brute force (finite differences).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle


def _one_query_attention(scores, values, scale=1.0):
    """Feed raw scores to the oracle: with one-hot keys K = I (d = N) the score
    of key j is scale * q[j], so q = scores / scale.  V is [N, d] padded to d = N
    columns with zeros."""
    s = np.asarray(scores, dtype=np.float64)
    n = len(s)
    vals = np.asarray(values, dtype=np.float64).reshape(n, -1)
    d = max(n, vals.shape[1])
    q = np.zeros((1, 1, n, d))
    q[0, 0, :, :n] = s / scale  # every query row asks the same question
    k = np.zeros((1, 1, n, d))
    k[0, 0, :, :n] = np.eye(n)
    v = np.zeros((1, 1, n, d))
    v[0, 0, :, : vals.shape[1]] = vals
    o, lse = oracle.attention_fwd(q, k, v, scale, False)
    return o[0, 0, 0, : vals.shape[1]], lse[0, 0, 0]


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked examples

def test_four_key_example_output(golden_dir):
    g = _load(golden_dir, "four_key_example.json")
    o, lse = _one_query_attention(g["scores"], g["values"])
    assert abs(o[0] - g["o"]["value"]) <= g["o"]["tol"]
    # the printed l is relative to the row maximum 5
    m = max(g["scores"])
    assert abs(math.exp(lse - m) - g["l"]["value"]) <= g["l"]["tol"]
    # o~ = o * l
    assert abs(o[0] * math.exp(lse - m) - g["o_tilde"]["value"]) <= g["o_tilde"]["tol"]


def test_four_key_example_weights(golden_dir):
    g = _load(golden_dir, "four_key_example.json")
    n = len(g["scores"])
    p, lse = _one_query_attention(g["scores"], np.eye(n))  # V = I exposes the weights
    m = max(g["scores"])
    w = p * math.exp(lse - m)  # weights relative to the maximum, as printed
    np.testing.assert_allclose(w, g["weights_rel_max"]["value"], atol=g["weights_rel_max"]["tol"])


def test_eight_score_example_running_sums(golden_dir):
    g = _load(golden_dir, "eight_score_example.json")
    seen = []
    for blk, m_exp, l_exp in zip(g["blocks"], g["running_max"], g["running_sum"]):
        seen += blk
        _, lse = _one_query_attention(seen, np.zeros(len(seen)))
        assert max(seen) == m_exp
        assert abs(math.exp(lse - m_exp) - l_exp) <= g["tol_sum"]


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_value_and_score():
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((2, 3, 1, 8)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, 0.5, causal)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, 0.5 * np.sum(q * k, axis=-1), rtol=1e-14, atol=1e-15)


def test_zero_keys_give_column_means():
    rng = np.random.default_rng(2)
    N, d = 37, 16
    q = rng.standard_normal((1, 2, N, d))
    k = np.zeros((1, 2, N, d))
    v = rng.standard_normal((1, 2, N, d))
    o, lse = oracle.attention_fwd(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-14)
    o, lse = oracle.attention_fwd(q, k, v, 0.3, True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-13)


def test_causal_first_row_is_first_value():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((1, 1, 9, 4)) for _ in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 1.0, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    assert abs(lse[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-14


def test_two_key_hand_example_logistic_weights():
    """d = 2, scale = 1, q0 = (1, 0), q1 = (0, 2), k0 = (3, 1), k1 = (1, 1):
    by hand S = [[3, 1], [2, 2]].  Row 0 weighs key 0 by the logistic
    1/(1+e^-2); row 1 splits evenly.  A transposed score matrix
    [[3, 2], [1, 2]] would change row 0."""
    q = np.array([[1.0, 0.0], [0.0, 2.0]]).reshape(1, 1, 2, 2)
    k = np.array([[3.0, 1.0], [1.0, 1.0]]).reshape(1, 1, 2, 2)
    v = np.array([[10.0, -1.0], [20.0, 5.0]]).reshape(1, 1, 2, 2)
    o, lse = oracle.attention_fwd(q, k, v, 1.0, False)
    w0 = 1.0 / (1.0 + math.exp(-2.0))
    np.testing.assert_allclose(o[0, 0, 0], w0 * v[0, 0, 0] + (1 - w0) * v[0, 0, 1], atol=1e-13)
    np.testing.assert_allclose(o[0, 0, 1], 0.5 * (v[0, 0, 0] + v[0, 0, 1]), atol=1e-13)
    assert abs(lse[0, 0, 0] - (3.0 + math.log1p(math.exp(-2.0)))) < 1e-13
    assert abs(lse[0, 0, 1] - (2.0 + math.log(2.0))) < 1e-13
    # causal: row 0 sees key 0 only, row 1 both
    o, lse = oracle.attention_fwd(q, k, v, 1.0, True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(lse[0, 0, 0] - 3.0) < 1e-14


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one_and_weights_are_exp_s_minus_lse(causal):
    """With one-hot keys S = scale * Q is known without a matmul; with V = I the
    output row is the softmax row itself."""
    rng = np.random.default_rng(4)
    N, scale = 24, 0.7
    q = rng.standard_normal((1, 1, N, N)) * 3
    k = np.eye(N).reshape(1, 1, N, N)
    v = np.eye(N).reshape(1, 1, N, N)
    p, lse = oracle.attention_fwd(q, k, v, scale, causal)
    p = p[0, 0]
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    s = scale * q[0, 0]
    if causal:
        s = np.where(np.tril(np.ones((N, N))) > 0, s, -np.inf)
        assert np.all(p[np.triu_indices(N, 1)] == 0.0)
    np.testing.assert_allclose(p, np.exp(s - lse[0, 0][:, None]), rtol=1e-13, atol=1e-16)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariance(causal):
    """Append one dimension with q = c_i / scale and k = 1: every score of row i
    gains c_i.  O must not change and LSE must shift by exactly c_i."""
    rng = np.random.default_rng(5)
    B, H, N, d, scale = 1, 2, 33, 8, 0.25
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    c = rng.uniform(-50, 50, size=(B, H, N))
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, N, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    o2, lse2 = oracle.attention_fwd(q2, k2, v2, scale, causal)
    np.testing.assert_allclose(o2[..., :d], o, atol=1e-12)
    np.testing.assert_allclose(lse2 - c, lse, atol=1e-11)


def test_key_permutation_and_value_linearity():
    rng = np.random.default_rng(6)
    B, H, N, d = 1, 1, 20, 6
    q, k, v, v2 = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.4, False)
    perm = rng.permutation(N)
    op, lsep = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(op, o, atol=1e-13)
    np.testing.assert_allclose(lsep, lse, atol=1e-13)
    oa, _ = oracle.attention_fwd(q, k, v + 2.0 * v2, 0.4, False)
    ob, _ = oracle.attention_fwd(q, k, v2, 0.4, False)
    np.testing.assert_allclose(oa, o + 2.0 * ob, atol=1e-12)


def test_sampled_rows_equal_full_rows():
    rng = np.random.default_rng(7)
    B, H, N, d = 2, 2, 40, 8
    q, k, v = (rng.standard_normal((B, H, N, d)) for _ in range(3))
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, 0.35, causal)
        bh = np.array([0, 3, 1, 2, 3])
        rows = np.array([0, 39, 17, 5, 1])
        os_, ls_ = oracle.attention_fwd_rows(q, k, v, 0.35, causal, bh, rows)
        np.testing.assert_allclose(os_, o.reshape(B * H, N, d)[bh, rows], atol=1e-14)
        np.testing.assert_allclose(ls_, lse.reshape(B * H, N)[bh, rows], atol=1e-14)


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 50, 16), (2, 1, 129, 8)])
def test_forward_matches_torch_fp64_sdpa(causal, shape):
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal(shape) for _ in range(3))
    scale = 1.0 / math.sqrt(shape[-1])
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), is_causal=causal, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_fp64_autograd(causal):
    rng = np.random.default_rng(9)
    shape = (1, 2, 45, 8)
    q, k, v, do = (rng.standard_normal(shape) for _ in range(4))
    scale = 0.3
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (3, 2), (6, 4)])
def test_backward_central_differences(causal, N, d):
    """dQ, dK, dV of L = sum(O * dO) against central differences of the forward."""
    rng = np.random.default_rng(10 + N)
    q, k, v, do = (rng.standard_normal((1, 1, N, d)) for _ in range(4))
    scale = 0.8
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal)
        return float(np.sum(o * do))

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*q.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(num)))
        assert err <= 1e-6, (which, err)


def test_backward_head_subset_matches_full():
    rng = np.random.default_rng(11)
    q, k, v, do = (rng.standard_normal((2, 2, 30, 8)) for _ in range(4))
    full = oracle.attention_bwd(q, k, v, do, 0.5, True)
    sub = oracle.attention_bwd(q, k, v, do, 0.5, True, heads=[3, 0])
    for f, s in zip(full, sub):
        f = f.reshape(4, 30, 8)
        np.testing.assert_array_equal(s, f[[3, 0]])


# ---------------------------------------------------------------- tile counts

@pytest.mark.parametrize("n", [1, 2, 7, 64, 256])
def test_causal_tile_counts_closed_form(n):
    """N = n T with square tiles: full = skipped = n(n-1)/2, masked = n."""
    T = 128
    assert oracle.tile_counts(n * T, True, T, T) == (n * (n - 1) // 2, n, n * (n - 1) // 2)
    assert oracle.tile_counts(n * T, False, T, T) == (n * n, 0, 0)


def test_ragged_tile_counts_by_hand():
    # N = 4000 = 31 * 128 + 32: the last key tile of every query tile runs past N
    assert oracle.tile_counts(4000, False, 128, 128) == (31 * 32, 32, 0)
    # a single key: the one tile is masked (it runs past N), nothing skipped
    assert oracle.tile_counts(1, True, 128, 128) == (0, 1, 0)
    # N = 129, causal: query tile 0 (rows 0..127) sees key tile 0 (diagonal,
    # masked) and skips tile 1 (j0 = 128 > 127); query tile 1 (row 128) sees
    # tile 0 fully and tile 1 (ragged, masked)
    assert oracle.tile_counts(129, True, 128, 128) == (1, 2, 1)
    # rectangular tiles, N = 256, causal, 128-row query tiles and 64-key tiles:
    # query tile 0: key tiles 0,1 masked (cross the diagonal), 2,3 skipped;
    # query tile 1: key tiles 0,1 full, 2,3 masked
    assert oracle.tile_counts(256, True, 128, 64) == (2, 4, 2)


# ---------------------------------------------------------------- packed variable-length batches

def _packed(seed, lens, H=2, d=16):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q, k, v, do = (rng.standard_normal((H, T, d)) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q, k, v, do, cu


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equal_lengths_is_the_dense_batch(causal):
    """B sequences of one length N packed head-major are the dense [B,H,N,d]
    batch with the batch and head axes swapped."""
    B, H, N, d = 3, 2, 37, 16
    q, k, v, do, cu = _packed(11, [N] * B, H, d)
    dense = lambda x: np.ascontiguousarray(x.reshape(H, B, N, d).transpose(1, 0, 2, 3))
    o, lse = oracle.attention_fwd_varlen(q, k, v, cu, 0.3, causal)
    o_d, lse_d = oracle.attention_fwd(dense(q), dense(k), dense(v), 0.3, causal)
    np.testing.assert_array_equal(o.reshape(H, B, N, d).transpose(1, 0, 2, 3), o_d)
    np.testing.assert_array_equal(lse.reshape(H, B, N).transpose(1, 0, 2), lse_d)
    g = oracle.attention_bwd_varlen(q, k, v, do, cu, 0.3, causal)
    g_d = oracle.attention_bwd(dense(q), dense(k), dense(v), dense(do), 0.3, causal)
    for a, b in zip(g, g_d):
        np.testing.assert_array_equal(a.reshape(H, B, N, d).transpose(1, 0, 2, 3), b)


def test_varlen_sequences_do_not_see_each_other():
    """Changing one sequence's keys and values leaves every other sequence's
    output and gradients unchanged, and changes its own."""
    lens = [5, 0, 17, 1, 9]
    q, k, v, do, cu = _packed(12, lens)
    o, lse = oracle.attention_fwd_varlen(q, k, v, cu, 0.25, True)
    g = oracle.attention_bwd_varlen(q, k, v, do, cu, 0.25, True)
    k2, v2 = k.copy(), v.copy()
    a, b = cu[2], cu[3]
    k2[:, a:b] += 1.0
    v2[:, a:b] *= -2.0
    o2, lse2 = oracle.attention_fwd_varlen(q, k2, v2, cu, 0.25, True)
    g2 = oracle.attention_bwd_varlen(q, k2, v2, do, cu, 0.25, True)
    outside = np.r_[0:a, b:cu[-1]]
    np.testing.assert_array_equal(o2[:, outside], o[:, outside])
    np.testing.assert_array_equal(lse2[:, outside], lse[:, outside])
    for x, y in zip(g, g2):
        np.testing.assert_array_equal(x[:, outside], y[:, outside])
    assert np.abs(o2[:, a:b] - o[:, a:b]).max() > 1e-3


def test_varlen_length_one_sequence_returns_its_value_row():
    """A sequence of one token attends only to itself: O = V, LSE = the scaled
    self-score (page "tm_flash_attention_math", "The problem": the single-query
    definition with one key)."""
    q, k, v, do, cu = _packed(13, [4, 1, 3])
    o, lse = oracle.attention_fwd_varlen(q, k, v, cu, 0.5, False)
    np.testing.assert_allclose(o[:, 4], v[:, 4], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, 4], 0.5 * np.einsum("hd,hd->h", q[:, 4], k[:, 4]), atol=1e-14)


# ---------------------------------------------------------------- decoding and block-state merge

@pytest.mark.parametrize("causal", [False, True])
def test_decode_rows_are_the_last_rows_of_full_attention(causal):
    """Queries at the end of a sequence: the decode oracle's rows equal the last
    Nq rows of the dense oracle run on the whole sequence (the C three-pass
    oracle; the decode oracle is numpy)."""
    rng = np.random.default_rng(21)
    B, H, Nkv, Nq, d = 2, 2, 57, 5, 16
    k, v = rng.standard_normal((B, H, Nkv, d)), rng.standard_normal((B, H, Nkv, d))
    q_full = rng.standard_normal((B, H, Nkv, d))
    o_full, lse_full = oracle.attention_fwd(q_full, k, v, 0.3, causal)
    o, lse = oracle.attention_fwd_decode(q_full[:, :, -Nq:], k, v, 0.3, causal)
    np.testing.assert_allclose(o, o_full[:, :, -Nq:], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_full[:, :, -Nq:], rtol=1e-12, atol=1e-13)


def test_decode_single_query_sees_every_key_when_causal():
    rng = np.random.default_rng(22)
    q, k, v = rng.standard_normal((1, 3, 1, 8)), rng.standard_normal((1, 3, 40, 8)), rng.standard_normal((1, 3, 40, 8))
    a = oracle.attention_fwd_decode(q, k, v, 0.5, True)
    b = oracle.attention_fwd_decode(q, k, v, 0.5, False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def _range_states(q, k, v, scale, bounds):
    """Per key range [a, b): that range's normalised output and log-sum-exp."""
    os_, ls_ = [], []
    for a, b in bounds:
        o, lse = oracle.attention_fwd_decode(q, k[:, :, a:b], v[:, :, a:b], scale, False)
        os_.append(o.reshape(-1, q.shape[-1]))
        ls_.append(lse.reshape(-1))
    return np.stack(os_), np.stack(ls_)


@pytest.mark.parametrize("bounds", [[(0, 10), (10, 57)], [(0, 1), (1, 2), (2, 30), (30, 57)],
                                    [(30, 57), (0, 30)]])
def test_merged_key_ranges_give_full_attention(bounds):
    """Exactness of the block-wise update ("Proof of exactness"): merging the
    states of disjoint key ranges, in any order, gives attention over all keys."""
    rng = np.random.default_rng(23)
    q, k, v = rng.standard_normal((1, 2, 3, 16)), rng.standard_normal((1, 2, 57, 16)), rng.standard_normal((1, 2, 57, 16))
    o_ref, lse_ref = oracle.attention_fwd_decode(q, k, v, 0.4, False)
    o, lse = oracle.merge_partials(*_range_states(q, k, v, 0.4, bounds))
    np.testing.assert_allclose(o, o_ref.reshape(-1, 16), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref.reshape(-1), rtol=1e-12, atol=1e-13)


def test_merge_ignores_ranges_without_visible_keys():
    rng = np.random.default_rng(24)
    o_part = rng.standard_normal((3, 4, 8))
    lse_part = rng.standard_normal((3, 4))
    lse_part[1] = -np.inf                       # range 1 saw no key for any row
    o_part[1] = 0.0
    a = oracle.merge_partials(o_part, lse_part)
    b = oracle.merge_partials(o_part[[0, 2]], lse_part[[0, 2]])
    np.testing.assert_allclose(a[0], b[0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-14, atol=1e-15)
    none = oracle.merge_partials(o_part[1:2], lse_part[1:2])
    assert np.all(none[0] == 0.0) and np.all(none[1] == -np.inf)
