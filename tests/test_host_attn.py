"""The host-CPU flash-style forward (libfattn_host) against the fp64 oracle.

The library runs the online-softmax recurrence in fp32 over 64-query tiles and
64-key blocks ("tm_flash_attention_math", "Why the same math matters on a
CPU"); the oracle materialises S and takes the three-pass softmax.  These
tests run on the CPU (no GPU marker).

Tolerances come from fp32 rounding: a score of d products carries a relative
error of order sqrt(d) * 2^-24 (about 1e-6 at d = 128), which is what O and
LSE show for N(0, 1) inputs; the bound is 20 times that, 2e-5.  With the
logit-stress distribution (Q ~ 4 N(0, 1)) scores are four times larger and
the bound is 1e-4.  A dropped rescale, a mask applied after the block max or
a per-block normalisation all produce errors of order 1e-1.
"""
import numpy as np
import pytest

import oracle
from online_softmax_08_gb300 import build as fbuild
from online_softmax_08_gb300 import fattn_host
from online_softmax_08_gb300.inputs import (HOST_WORKLOADS, default_scale, make_host_inputs,
                                            sample_rows)

TOL = {1.0: 2e-5, 4.0: 1e-4}


@pytest.fixture(scope="module", autouse=True)
def lib():
    fbuild.build_host()
    return fattn_host.load()


def _f64(*xs):
    return tuple(x.astype(np.float64) for x in xs)


def _check(o, lse, o_ref, lse_ref, tol):
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(o - o_ref).max() <= tol
    assert np.abs(lse - lse_ref).max() <= tol


CASES = [
    # B, H, N, d, causal, q_std, v_dist: several tiles, ragged tails, every d path
    (2, 3, 200, 64, True, 1.0, "normal"),
    (2, 3, 200, 64, False, 1.0, "normal"),
    (1, 2, 130, 128, True, 1.0, "normal"),
    (1, 2, 129, 128, False, 1.0, "normal"),
    (1, 1, 77, 40, False, 1.0, "normal"),    # d not a multiple of 16
    (1, 1, 65, 1, True, 1.0, "normal"),      # d = 1
    (1, 1, 300, 256, True, 1.0, "normal"),   # largest d
    (1, 2, 333, 128, False, 4.0, "uniform"),  # logit stress, ragged
    (1, 2, 700, 64, True, 4.0, "uniform"),
    (3, 1, 64, 64, True, 1.0, "normal"),     # exactly one tile
]


@pytest.mark.parametrize("B,H,N,d,causal,q_std,v_dist", CASES)
def test_forward_matches_oracle(B, H, N, d, causal, q_std, v_dist):
    q, k, v = make_host_inputs(B, H, N, d, 71 + N + d, q_std, v_dist)
    scale = default_scale(d)
    o, lse = fattn_host.forward(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.attention_fwd(*_f64(q, k, v), scale, causal)
    _check(o, lse, o_ref, lse_ref, TOL[q_std])


def test_single_key_returns_v():
    # N = 1: the only weight is 1, so O = V exactly and LSE is the one score
    q, k, v = make_host_inputs(2, 2, 1, 64, 5)
    o, lse = fattn_host.forward(q, k, v, 0.125, True)
    assert np.array_equal(o, v)
    s = 0.125 * np.sum(q.astype(np.float64) * k, axis=-1)
    assert np.abs(lse - s).max() <= 2e-6


@pytest.mark.parametrize("causal", [False, True])
def test_zero_keys_give_prefix_means(causal):
    # K = 0: every visible score is 0, so O_i is the mean of the visible V rows
    # and LSE_i = ln(count)
    N, d = 150, 64
    q, _, v = make_host_inputs(1, 1, N, d, 6)
    k = np.zeros_like(q)
    o, lse = fattn_host.forward(q, k, v, 0.125, causal)
    vv = v[0, 0].astype(np.float64)
    if causal:
        count = np.arange(1, N + 1, dtype=np.float64)
        mean = np.cumsum(vv, axis=0) / count[:, None]
    else:
        count = np.full(N, float(N))
        mean = np.broadcast_to(vv.mean(axis=0), (N, d))
    assert np.abs(o[0, 0] - mean).max() <= 2e-6
    assert np.abs(lse[0, 0] - np.log(count)).max() <= 2e-6


def test_huge_logits_stay_finite():
    # scores near 2000: every exponent is <= 0, nothing overflows.  A score
    # carries an fp32 error of about sqrt(d) 2^-24 of its size, which moves the
    # weights, and so O, by about that much: the bound scales with max |S|.
    q, k, v = make_host_inputs(1, 2, 190, 64, 8, q_std=400.0)
    o, lse = fattn_host.forward(q, k, v, 0.125, True)
    o_ref, lse_ref = oracle.attention_fwd(*_f64(q, k, v), 0.125, True)
    s_max = np.abs(lse_ref).max()
    assert s_max > 1000 and np.isfinite(o).all()
    assert np.abs(o - o_ref).max() <= 4e-7 * s_max + 2e-5
    assert np.abs(lse - lse_ref).max() <= 4e-7 * s_max + 2e-5


def test_result_is_independent_of_thread_count():
    q, k, v = make_host_inputs(1, 5, 333, 128, 9)
    ref = fattn_host.forward(q, k, v, 0.09, True, n_threads=1)
    for nt in (2, 3, 0):
        o, lse = fattn_host.forward(q, k, v, 0.09, True, n_threads=nt)
        assert np.array_equal(o, ref[0]) and np.array_equal(lse, ref[1])


def test_empty_problems():
    for shape in ((1, 1, 0, 64), (0, 2, 10, 64), (2, 0, 10, 64)):
        q = np.zeros(shape, np.float32)
        o, lse = fattn_host.forward(q, q, q, 0.1, True)
        assert o.shape == shape and lse.shape == shape[:3]


def test_argument_errors():
    q = np.zeros((1, 1, 8, 16), np.float32)
    o, lse = np.zeros_like(q), np.zeros((1, 1, 8), np.float32)
    lib = fattn_host.load()
    P = q.ctypes.data
    call = lambda *a: lib.fattn_host_fwd(*a)
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 16, 0.1, 1, 0) == 0
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 0, 0.1, 1, 0) == 2
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 257, 0.1, 1, 0) == 2
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 16, 0.0, 1, 0) == 1
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 16, float("nan"), 1, 0) == 1
    assert call(P, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, -1, 16, 0.1, 1, 0) == 1
    assert call(None, P, P, o.ctypes.data, lse.ctypes.data, 1, 1, 8, 16, 0.1, 1, 0) == 1
    assert call(P, P, P, o.ctypes.data, None, 1, 1, 8, 16, 0.1, 1, 0) == 1
    with pytest.raises(TypeError):
        fattn_host.forward(q.astype(np.float64), q, q, 0.1, True)


def test_exp2_within_one_and_a_half_ulp():
    # the library's exp2 (range reduction + degree-7 Taylor polynomial of 2^f)
    # against fp64 exp2 over its whole domain (0.83 ulp at most with fused
    # multiply-adds, 1.1 without); integers map to exact powers of 2
    rng = np.random.default_rng(0)
    t = np.concatenate([np.linspace(-126.0, 0.0, 400_001), -126.0 * rng.random(400_000),
                        -rng.random(100_000)]).astype(np.float32)
    y = fattn_host.exp2(t).astype(np.float64)
    ref = np.exp2(t.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert (np.abs(y - ref) / ulp).max() <= 1.5
    ints = -np.arange(0, 127, dtype=np.float32)
    assert np.array_equal(fattn_host.exp2(ints), np.exp2(ints))
    assert np.array_equal(fattn_host.exp2(np.array([-127.0, -200.0, -np.inf], np.float32)),
                          np.zeros(3, np.float32))


def test_fma_peak_is_positive_and_bounds_the_forward():
    import time
    peak = fattn_host.fma_peak_gflops(0, 0.2)
    assert peak > 0
    q, k, v = make_host_inputs(1, 4, 1024, 64, 10)
    fattn_host.forward(q, k, v, 0.125, False)
    t0 = time.perf_counter()
    fattn_host.forward(q, k, v, 0.125, False)
    gflops = 4 * 4 * 1024 * 1024 * 64 / (time.perf_counter() - t0) / 1e9
    assert gflops < 1.25 * peak


@pytest.mark.parametrize("name", sorted(HOST_WORKLOADS))
def test_host_workload_sampled_rows(name):
    # the benchmarked shape, in full, checked on seeded rows of four heads
    w = HOST_WORKLOADS[name]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v = make_host_inputs(B, H, N, d, w["seed"])
    scale = default_scale(d)
    o, lse = fattn_host.forward(q, k, v, scale, w["causal"])
    rng = np.random.default_rng(w["seed"])
    heads = rng.choice(B * H, size=min(4, B * H), replace=False)
    rows = sample_rows(N, 48, w["seed"])
    bh = np.repeat(heads, len(rows))
    rr = np.tile(rows, len(heads))
    o_ref, lse_ref = oracle.attention_fwd_rows(*_f64(q, k, v), scale, w["causal"], bh, rr)
    _check(o.reshape(B * H, N, d)[bh, rr], lse.reshape(B * H, N)[bh, rr], o_ref, lse_ref,
           TOL[1.0])
