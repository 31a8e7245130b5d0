"""fattn_fwd_bwd_host: forward + backward of host-resident tensors, staged
through the device in chunks of heads with copies and kernels overlapped.

Each (b, h) slice is an independent problem, so a chunked run must give what
fattn_fwd + fattn_bwd give on the whole tensor: O, LSE, dK and dV bit for bit
(their kernels reduce in a fixed order), and dQ up to the order of its fp32
partial-sum reductions (within one bf16 rounding step).  The small cases are
also checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import WORKLOADS, default_scale, make_inputs

pytestmark = pytest.mark.gpu


def _device_reference(q, k, v, do, scale, causal):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fattn.forward(qd, kd, vd, scale, causal)
    dq, dk, dv = fattn.backward(qd, kd, vd, o, lse, dod, scale, causal)
    torch.cuda.synchronize()
    return tuple(x.cpu() for x in (o, lse, dq, dk, dv))


def _staged(q, k, v, do, scale, causal, heads, pin=True):
    if pin:
        q, k, v, do = (x.pin_memory() for x in (q, k, v, do))
    out = fattn.forward_backward_host(q, k, v, do, scale, causal, heads_per_chunk=heads)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    return out


def _same_as_device(got, ref):
    o, lse, dq, dk, dv = got
    ro, rlse, rdq, rdk, rdv = ref
    assert torch.equal(o, ro) and torch.equal(lse, rlse)
    assert torch.equal(dk, rdk) and torch.equal(dv, rdv)
    a, b = dq.float(), rdq.float()
    assert ((a - b).abs() <= a.abs().maximum(b.abs()) * 2.0 ** -7 + 1e-6).all()


def _against_oracle(q, k, v, do, scale, causal, got):
    f64 = lambda t: t.to(torch.float64).numpy()
    o_ref, lse_ref = oracle.attention_fwd(f64(q), f64(k), f64(v), scale, causal)
    assert np.abs(f64(got[0]) - o_ref).max() <= 2e-2
    assert np.abs(f64(got[1]) - lse_ref).max() <= 1e-3
    for g, r in zip(got[2:], oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), scale, causal)):
        err = np.abs(f64(g) - r)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


@pytest.mark.parametrize("B,H,N,d,causal,heads", [
    (1, 5, 300, 64, True, 2),      # three chunks, the last one ragged
    (2, 4, 1024, 128, False, 1),   # eight chunks: every slot reused
    (1, 3, 129, 128, True, 0),     # the library's chunk size
    (2, 2, 200, 64, False, 7),     # one chunk larger than B*H
])
def test_staged_matches_device_api_and_oracle(B, H, N, d, causal, heads):
    q, k, v, do = make_inputs(B, H, N, d, seed=300 + N, with_do=True)
    scale = default_scale(d)
    got = _staged(q, k, v, do, scale, causal, heads)
    _same_as_device(got, _device_reference(q, k, v, do, scale, causal))
    _against_oracle(q, k, v, do, scale, causal, got)


def test_pageable_host_memory_gives_the_same_results():
    q, k, v, do = make_inputs(1, 4, 256, 64, seed=310, with_do=True)
    got = _staged(q, k, v, do, 0.125, True, 1, pin=False)
    _same_as_device(got, _device_reference(q, k, v, do, 0.125, True))


def test_ordered_on_the_callers_stream():
    # results are complete once the caller's stream is synchronised, and a
    # second call on another stream with its own workspace does not disturb them
    q, k, v, do = (x.pin_memory() for x in make_inputs(1, 6, 512, 128, seed=311, with_do=True))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        a = fattn.forward_backward_host(q, k, v, do, 0.09, True, heads_per_chunk=2, stream=s1)
    with torch.cuda.stream(s2):
        b = fattn.forward_backward_host(q, k, v, do, 0.09, True, heads_per_chunk=3, stream=s2)
    s1.synchronize()
    s2.synchronize()
    for x, y in zip(a[:2], b[:2]):
        assert torch.equal(x, y)
    _same_as_device(a, _device_reference(q.clone(), k.clone(), v.clone(), do.clone(), 0.09, True))


def test_headline_size_matches_device_api():
    w = WORKLOADS["b1h32_n8192_d128_causal"]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v, do = make_inputs(B, H, N, d, w["seed"], with_do=True)
    scale = default_scale(d)
    got = _staged(q, k, v, do, scale, True, 0)
    _same_as_device(got, _device_reference(q, k, v, do, scale, True))
