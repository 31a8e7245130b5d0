"""Forward parity: libfattn's sm_103a kernel against the fp64 oracle.

Bar (from the workload definition): O max-abs <= 2e-2 and mean-abs <= 2e-3,
LSE <= 1e-3 absolute, tile counts exact.  Small problems are compared element
by element; the full-size workloads are run in the launch configuration the
benchmark times and compared on seeded samples of query rows, each row
computed by the oracle one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import WORKLOADS, default_scale, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _run(q, k, v, scale, causal, counts=False):
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev).contiguous() for x in (q, k, v))
    tc = torch.zeros(3, dtype=torch.int64, device=dev) if counts else None
    o, lse = fattn.forward(qd, kd, vd, scale, causal, tile_counts=tc)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    return o, lse, (tc.cpu().tolist() if counts else None)


def _check(o_gpu, lse_gpu, o_ref, lse_ref):
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    assert np.abs(lse_gpu - lse_ref).max() <= LSE_MAX, np.abs(lse_gpu - lse_ref).max()


def _expected_counts(B, H, N, d, causal):
    bq, bk = fattn.fattn_tile_sizes(d, 0)
    full, masked, skipped = oracle.tile_counts(N, causal, bq, bk)
    return [B * H * full, B * H * masked, B * H * skipped]


# ---------------------------------------------------------------- element by element

SMALL = [
    # (B, H, N, d, causal)  -- several tiles, ragged tails, the degenerate sizes
    (1, 1, 256, 64, False),   # the single-head workload
    (1, 2, 300, 128, False),
    (1, 2, 300, 128, True),
    (2, 1, 129, 64, True),
    (1, 1, 1, 128, False),
    (1, 1, 1, 64, True),
    (1, 3, 127, 128, True),
    (1, 1, 128, 64, True),
    (2, 2, 513, 128, True),
    (1, 2, 1000, 64, False),
    (1, 1, 640, 128, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_forward_matches_oracle_elementwise(B, H, N, d, causal):
    q, k, v = make_inputs(B, H, N, d, seed=4242 + N + d)
    scale = default_scale(d)
    o, lse, counts = _run(q, k, v, scale, causal, counts=True)
    o_ref, lse_ref = oracle.attention_fwd(_f64(q), _f64(k), _f64(v), scale, causal)
    _check(_f64(o), _f64(lse), o_ref, lse_ref)
    assert counts == _expected_counts(B, H, N, d, causal)


def test_single_head_workload_full():
    w = WORKLOADS["single_head_n256_d64"]
    q, k, v = make_inputs(w["B"], w["H"], w["N"], w["d"], w["seed"])
    scale = default_scale(w["d"])
    o, lse, _ = _run(q, k, v, scale, False)
    o_ref, lse_ref = oracle.attention_fwd(_f64(q), _f64(k), _f64(v), scale, False)
    _check(_f64(o), _f64(lse), o_ref, lse_ref)


def test_logit_stress_small_elementwise():
    """Scores with standard deviation 4 and a ragged last tile: the running
    maximum rises late and alpha rescaling is exercised on every row."""
    q, k, v = make_inputs(1, 2, 600, 128, seed=77, q_std=4.0, v_dist="uniform")
    scale = default_scale(128)
    o, lse, _ = _run(q, k, v, scale, False)
    o_ref, lse_ref = oracle.attention_fwd(_f64(q), _f64(k), _f64(v), scale, False)
    _check(_f64(o), _f64(lse), o_ref, lse_ref)


def test_extreme_logits_do_not_overflow():
    """Scores far beyond exp's fp32 range (the stability claim of
    tm_flash_attention_math, "Proof of numerical stability")."""
    q, k, v = make_inputs(1, 1, 384, 64, seed=78)
    q = (q.float() * 60.0).to(torch.bfloat16)
    scale = default_scale(64)
    o, lse, _ = _run(q, k, v, scale, True)
    o_ref, lse_ref = oracle.attention_fwd(_f64(q), _f64(k), _f64(v), scale, True)
    assert np.isfinite(_f64(o)).all()
    _check(_f64(o), _f64(lse), o_ref, lse_ref)


def test_repeated_calls_are_deterministic():
    q, k, v = make_inputs(1, 4, 700, 128, seed=79)
    o1, l1, _ = _run(q, k, v, 0.1, True)
    o2, l2, _ = _run(q, k, v, 0.1, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ---------------------------------------------------------------- full-size workloads

def _sampled(name, causal, n_rows=64, n_heads=4):
    w = WORKLOADS[name]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v = make_inputs(B, H, N, d, w["seed"], w["q_std"], w["v_dist"])
    scale = default_scale(d)
    o, lse, counts = _run(q, k, v, scale, causal, counts=True)
    assert counts == _expected_counts(B, H, N, d, causal)
    g = torch.Generator().manual_seed(w["seed"])
    heads = torch.randperm(B * H, generator=g)[:n_heads].tolist()
    rows = sample_rows(N, n_rows, w["seed"])
    bh = np.repeat(heads, len(rows))
    rr = np.tile(rows, len(heads))
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    o_ref, lse_ref = oracle.attention_fwd_rows(qf, kf, vf, scale, causal, bh, rr)
    o_gpu = _f64(o).reshape(B * H, N, d)[bh, rr]
    lse_gpu = _f64(lse).reshape(B * H, N)[bh, rr]
    _check(o_gpu, lse_gpu, o_ref, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_b4h16_n2048_d64_sampled(causal):
    _sampled("b4h16_n2048_d64", causal)


def test_headline_b1h32_n8192_d128_causal_sampled():
    _sampled("b1h32_n8192_d128_causal", True)


def test_logit_stress_b2h16_n4000_d128_sampled():
    _sampled("logit_stress_b2h16_n4000_d128", False)


def test_long_b1h16_n32768_d128_causal_sampled():
    _sampled("long_b1h16_n32768_d128_causal", True, n_rows=64, n_heads=2)


# ---------------------------------------------------------------- argument checks

def test_invalid_arguments_launch_nothing():
    lib = fattn.load()
    dev = torch.device("cuda:0")
    x = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device=dev)
    p = x.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.fattn_fwd(None, p, p, p, lse.data_ptr(), 1, 1, 128, 128, 0.1, 0, s) == 1
    assert lib.fattn_fwd(p + 2, p, p, p, lse.data_ptr(), 1, 1, 128, 128, 0.1, 0, s) == 1
    assert lib.fattn_fwd(p, p, p, p, lse.data_ptr(), 1, 1, 128, 96, 0.1, 0, s) == 2
    assert lib.fattn_fwd(p, p, p, p, lse.data_ptr(), 1, 1, 0, 128, 0.1, 0, s) == 1
    assert lib.fattn_fwd(p, p, p, p, lse.data_ptr(), 1, 1, 128, 128, -1.0, 0, s) == 1
    assert lib.fattn_fwd(p, p, p, p, lse.data_ptr(), 1, 1, 128, 128, float("nan"), 0, s) == 1
    torch.cuda.synchronize()
