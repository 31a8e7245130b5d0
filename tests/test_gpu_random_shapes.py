"""Seeded sweep of shapes the fixed workloads do not cover: ragged N from 1 to
1100, batch and head counts of 1-3, both head sizes, both masks, and softmax
scales other than 1/sqrt(d) (the scale is an argument of the interface).  The
scaled scores keep a standard deviation between 0.5 and 1.5, the range the
2e-2 bars of the fixed workloads were set for (their scores have standard
deviation 1; sharper ones need the derived bars of the logit-stress tests).
Each case runs the forward (O, LSE, tile counts) and the backward (dQ, dK, dV)
and compares every element with the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3
G_MAX, G_MEAN = 2e-2, 2e-3


def _cases(count=24, seed=20261203):
    rng = np.random.RandomState(seed)
    out = []
    for i in range(count):
        B = int(rng.randint(1, 4))
        H = int(rng.randint(1, 4))
        N = int(rng.randint(1, 1101))
        d = int(rng.choice([64, 128]))
        causal = bool(rng.randint(0, 2))
        q_std = float(rng.choice([1.0, 1.5]))
        spread = float(rng.uniform(0.5, 1.5))  # standard deviation of the scaled scores
        scale = spread / (q_std * math.sqrt(d))
        out.append((B, H, N, d, causal, q_std, round(scale, 6), 7000 + i))
    return out


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _close(got, ref, bar_max, bar_mean, what):
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref)
    assert err.max() <= bar_max, (what, float(err.max()))
    assert err.mean() <= bar_mean, (what, float(err.mean()))


@pytest.mark.parametrize("B,H,N,d,causal,q_std,scale,seed", _cases())
def test_random_shape_forward_and_backward(B, H, N, d, causal, q_std, scale, seed):
    q, k, v, do = make_inputs(B, H, N, d, seed, q_std=q_std, with_do=True)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (x.to(dev).contiguous() for x in (q, k, v, do))
    tc = torch.zeros(3, dtype=torch.int64, device=dev)
    o, lse = fattn.forward(qd, kd, vd, scale, causal, tile_counts=tc)
    dq, dk, dv = fattn.backward(qd, kd, vd, o, lse, dod, scale, causal)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0

    qf, kf, vf, dof = _f64(q), _f64(k), _f64(v), _f64(do)
    o_ref, lse_ref = oracle.attention_fwd(qf, kf, vf, scale, causal)
    _close(_f64(o), o_ref, O_MAX, O_MEAN, "o")
    assert np.abs(_f64(lse) - lse_ref).max() <= LSE_MAX
    bq, bk = fattn.fattn_tile_sizes(d, 0)
    full, masked, skipped = oracle.tile_counts(N, causal, bq, bk)
    assert tc.cpu().tolist() == [B * H * full, B * H * masked, B * H * skipped]

    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv),
                              oracle.attention_bwd(qf, kf, vf, dof, scale, causal)):
        _close(_f64(got), ref, G_MAX, G_MEAN, name)
