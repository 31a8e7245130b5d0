"""The entry points can be captured into a CUDA graph and replayed: no host
synchronisation, allocation or device-wide call inside fattn_fwd, fattn_bwd,
fattn_decode or fattn_softmax_rows once each has run once on the device.
Replays give the eager results (bit for bit where the work has a fixed order;
dQ, added by atomic bulk reductions, to within rounding)."""
import pytest
import torch

from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_inputs

pytestmark = pytest.mark.gpu


def test_forward_backward_graph_replays_match_eager():
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 4, 1000, 128
    scale = default_scale(d)
    q, k, v, do = (x.to(dev) for x in make_inputs(B, H, N, d, seed=31, with_do=True))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fattn.fattn_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)

    def step(stream):
        fattn.fattn_fwd(q, k, v, o, lse, B, H, N, d, scale, True, stream)
        fattn.fattn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, True, ws, ws.numel(),
                        stream)

    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        step(s)                                  # eager run (first-use setup happens here)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    for got, want in zip((o, lse, dk, dv), (eager[0], eager[1], eager[3], eager[4])):
        assert torch.equal(got, want)
    assert (dq.float() - eager[2].float()).abs().max().item() <= 2e-3


def test_decode_and_softmax_graph_replays_match_eager():
    dev = torch.device("cuda:0")
    B, H, Nq, Nkv, d = 2, 4, 3, 2000, 64
    q, k, v = make_inputs(B, H, Nkv, d, seed=32)
    q = q[:, :, Nkv - Nq:].contiguous().to(dev)
    k, v = k.to(dev), v.to(dev)
    scale = default_scale(d)
    lib = fattn.load()
    ws = torch.empty(int(lib.fattn_decode_workspace_bytes(B, H, Nq, Nkv, d, 0)), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device=dev)
    x = torch.randn(64, 3000, generator=torch.Generator().manual_seed(33)).to(dev)
    y = torch.empty_like(x)
    s = torch.cuda.Stream(device=dev)

    def step():
        fattn._check("fattn_decode", lib.fattn_decode(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nkv, d,
            scale, 1, 0, ws.data_ptr(), ws.numel(), s.cuda_stream))
        fattn._check("fattn_softmax_rows", lib.fattn_softmax_rows(
            x.data_ptr(), y.data_ptr(), None, 64, 3000, s.cuda_stream))

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, y)]
    for t in (o, lse, y):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    g.replay()
    torch.cuda.synchronize()
    for got, want in zip((o, lse, y), eager):
        assert torch.equal(got, want)
