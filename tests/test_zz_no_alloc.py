"""fattn_bwd_noalloc: the backward pass with the library's built-in workspace.

It exists for callers that cannot allocate device memory where they run the
backward (a plugin inside a host program that owns the CUDA allocator, or a
runtime that reserves its whole memory budget up front).  This file runs last
(pytest collects it after the others), so a failure here does not hide any
other test when the run stops at the first failure; it also passes when run
alone in a fresh process.

Checks: two calls in a row through the C-ABI agree with fattn_bwd (the
entry point that takes a caller workspace) within the parity tolerance of the
other backward tests; a small call made right after a larger one (so the
array still holds the larger call's data) matches the fp64 oracle; a problem
whose workspace exceeds the built-in size is rejected before any launch.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_inputs

G_MAX, G_MEAN = 2e-2, 2e-3
SCRATCH_BYTES = 64 << 20  # FATTN_NOALLOC_SCRATCH_BYTES in include/fattn.h


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 777, 128, True), (2, 2, 640, 64, False)])
def test_noalloc_matches_workspace_backward_twice(B, H, N, d, causal):
    dev = torch.device("cuda:0")
    q, k, v, do = (x.to(dev) for x in make_inputs(B, H, N, d, seed=6060 + N, with_do=True))
    scale = default_scale(d)
    o, lse = fattn.forward(q, k, v, scale, causal)
    ref = fattn.backward(q, k, v, o, lse, do, scale, causal)
    lib = fattn.load()
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        status = lib.fattn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale,
                                       int(causal), s)
        assert status == 0, fattn.fattn_status_string(status)
        torch.cuda.synchronize()
        for got, want in zip((dq, dk, dv), ref):
            err = np.abs(_f64(got) - _f64(want))
            assert err.max() <= G_MAX and err.mean() <= G_MEAN
    assert fattn.fattn_device_error() == 0


def _noalloc(q, k, v, o, lse, do, scale, causal):
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    status = fattn.load().fattn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, int(causal),
        torch.cuda.current_stream().cuda_stream)
    assert status == 0, fattn.fattn_status_string(status)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_after_a_larger_call_matches_the_oracle():
    """A ragged small problem right after a large one that filled much of the
    array: the stale contents must not leak into the small call's results."""
    dev = torch.device("cuda:0")
    big = [x.to(dev) for x in make_inputs(1, 8, 4000, 128, seed=6161, with_do=True)]
    scale = default_scale(128)
    o, lse = fattn.forward(*big[:3], scale, True)
    _noalloc(*big[:3], o, lse, big[3], scale, True)
    q, k, v, do = make_inputs(1, 1, 777, 128, seed=6162, with_do=True)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fattn.forward(qd, kd, vd, scale, True)
    got = _noalloc(qd, kd, vd, o, lse, dod, scale, True)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    ref = oracle.attention_bwd(f64(q), f64(k), f64(v), f64(do), scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        err = np.abs(f64(g) - r)
        assert err.max() <= G_MAX and err.mean() <= G_MEAN, (name, err.max(), err.mean())


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_the_scratch_size():
    B, H, N, d = 1, 8, 16384, 128
    assert fattn.fattn_bwd_workspace_bytes(B, H, N, d) > SCRATCH_BYTES
    lib = fattn.load()
    a = 1 << 20  # never dereferenced: the size check comes first
    assert lib.fattn_bwd_noalloc(a, a, a, a, a, a, a, a, a, B, H, N, d, 0.1, 1, None) == 4
