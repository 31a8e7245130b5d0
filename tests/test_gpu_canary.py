"""Canary tests: no entry point writes outside the buffers it was given.

Every output (and every workspace) below is an interior view of a larger buffer
whose bytes were all set to a sentinel.  After the call the bytes before and
after the interior must still hold the sentinel.  The shapes are the ones where
a tile, a row or a sequence ends inside a tile: ragged N, sequences of length 0,
1 and 129, a single query, rows that do not fill a vector.
"""
import pytest
import torch

from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_inputs, make_varlen_inputs

pytestmark = pytest.mark.gpu

SENT = 0x5A
PAD = 4096  # bytes on each side; keeps every interior 256-byte aligned
DEV = torch.device("cuda:0")


class Guarded:
    """A tensor of `shape` and `dtype` inside a sentinel-filled byte buffer."""

    def __init__(self, shape, dtype, device=DEV, pin=False, nbytes=None):
        elem = torch.empty((), dtype=dtype).element_size()
        numel = 1
        for s in shape:
            numel *= s
        self.n = numel * elem if nbytes is None else nbytes
        buf = torch.full((self.n + 2 * PAD,), SENT, dtype=torch.uint8, device=device)
        self.buf = buf.pin_memory() if pin else buf
        inner = self.buf[PAD:PAD + self.n]
        self.t = inner.view(dtype)[:numel].view(shape) if nbytes is None else inner

    def intact(self):
        head, tail = self.buf[:PAD], self.buf[PAD + self.n:]
        return bool((head == SENT).all()) and bool((tail == SENT).all())


def _sync_ok():
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0


@pytest.mark.parametrize("B,H,N,d,causal", [
    (1, 2, 300, 128, True), (1, 1, 129, 64, False), (2, 1, 1, 128, True), (1, 1, 4000, 128, False),
])
def test_forward_and_backward_stay_inside_their_buffers(B, H, N, d, causal):
    q, k, v, do = (x.to(DEV) for x in make_inputs(B, H, N, d, seed=500 + N, with_do=True))
    scale = default_scale(d)
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    counts = Guarded((3,), torch.int64)
    counts.t.zero_()
    fattn.fattn_fwd_ex(q, k, v, o.t, lse.t, B, H, N, d, scale, causal, counts.t)
    _sync_ok()
    assert o.intact() and lse.intact() and counts.intact()
    o_ref, lse_ref = fattn.forward(q, k, v, scale, causal)
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_ref) and torch.equal(lse.t, lse_ref)

    grads = [Guarded((B, H, N, d), torch.bfloat16) for _ in range(3)]
    wsb = fattn.fattn_bwd_workspace_bytes(B, H, N, d)
    ws = Guarded((wsb,), torch.uint8)
    fattn.fattn_bwd(q, k, v, o.t, lse.t, do, grads[0].t, grads[1].t, grads[2].t, B, H, N, d, scale,
                    causal, ws.t, wsb)
    _sync_ok()
    assert all(g.intact() for g in grads) and ws.intact()


def test_varlen_stays_inside_its_buffers():
    lengths, H, d = [1, 127, 300, 0, 129], 2, 128
    q, k, v, do, cu = make_varlen_inputs(lengths, H, d, seed=510, with_do=True)
    q, k, v, do, cu = (x.to(DEV) for x in (q, k, v, do, cu))
    T, B, mx = q.shape[1], len(lengths), max(lengths)
    scale = default_scale(d)
    o = Guarded((H, T, d), torch.bfloat16)
    lse = Guarded((H, T), torch.float32)
    fattn.fattn_fwd_varlen(q, k, v, o.t, lse.t, cu, B, H, mx, T, d, scale, True)
    _sync_ok()
    assert o.intact() and lse.intact()
    grads = [Guarded((H, T, d), torch.bfloat16) for _ in range(3)]
    wsb = fattn.fattn_bwd_workspace_bytes(1, H, T, d)
    ws = Guarded((wsb,), torch.uint8)
    fattn.fattn_bwd_varlen(q, k, v, o.t, lse.t, do, grads[0].t, grads[1].t, grads[2].t, cu, B, H,
                           mx, T, d, scale, True, ws.t, wsb)
    _sync_ok()
    assert all(g.intact() for g in grads) and ws.intact()


@pytest.mark.parametrize("splits", [0, 3])
def test_decode_and_merge_stay_inside_their_buffers(splits):
    B, H, Nq, Nkv, d = 1, 2, 3, 1000, 128
    q, _, _ = make_inputs(B, H, Nq, d, seed=520)
    _, k, v = make_inputs(B, H, Nkv, d, seed=521)
    q, k, v = (x.to(DEV) for x in (q, k, v))
    lib = fattn.load()
    o = Guarded((B, H, Nq, d), torch.bfloat16)
    lse = Guarded((B, H, Nq), torch.float32)
    wsb = int(lib.fattn_decode_workspace_bytes(B, H, Nq, Nkv, d, splits))
    ws = Guarded((max(wsb, 1),), torch.uint8)
    fattn._check("fattn_decode", lib.fattn_decode(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.t.data_ptr(), lse.t.data_ptr(), B, H, Nq, Nkv,
        d, default_scale(d), 1, splits, ws.t.data_ptr(), wsb,
        torch.cuda.current_stream().cuda_stream))
    _sync_ok()
    assert o.intact() and lse.intact() and ws.intact()

    S, rows = 3, 7
    g = torch.Generator(device="cpu").manual_seed(522)
    o_part = torch.randn((S, rows, d), generator=g).to(DEV)
    lse_part = torch.randn((S, rows), generator=g).to(DEV)
    om = Guarded((rows, d), torch.bfloat16)
    lm = Guarded((rows,), torch.float32)
    fattn._check("fattn_merge_partials", lib.fattn_merge_partials(
        o_part.data_ptr(), lse_part.data_ptr(), S, rows, d, om.t.data_ptr(), lm.t.data_ptr(),
        torch.cuda.current_stream().cuda_stream))
    _sync_ok()
    assert om.intact() and lm.intact()


@pytest.mark.parametrize("rows,cols", [(5, 1000), (3, 1001), (2, 50001), (1, 1)])
def test_row_softmax_stays_inside_its_buffers(rows, cols):
    # 16-byte rows, rows that are not, and rows longer than the shared-memory staging
    g = torch.Generator(device="cpu").manual_seed(530 + cols)
    x = (torch.randn((rows, cols), generator=g) * 10.0).to(DEV)
    y = Guarded((rows, cols), torch.float32)
    lse = Guarded((rows,), torch.float32)
    fattn._check("fattn_softmax_rows", fattn.load().fattn_softmax_rows(
        x.data_ptr(), y.t.data_ptr(), lse.t.data_ptr(), rows, cols,
        torch.cuda.current_stream().cuda_stream))
    _sync_ok()
    assert y.intact() and lse.intact()
    assert torch.allclose(y.t, torch.softmax(x, dim=1), atol=1e-6, rtol=1e-5)


def test_host_staged_path_stays_inside_its_buffers():
    B, H, N, d = 1, 3, 200, 64
    host = [x.pin_memory() for x in make_inputs(B, H, N, d, seed=540, with_do=True)]
    outs = [Guarded((B, H, N, d), torch.bfloat16, device="cpu", pin=True) for _ in range(4)]
    lse = Guarded((B, H, N), torch.float32, device="cpu", pin=True)
    wsb = fattn.fattn_fwd_bwd_host_workspace_bytes(B, H, N, d, 2)
    ws = Guarded((wsb,), torch.uint8)
    fattn.fattn_fwd_bwd_host(*host, outs[0].t, lse.t, outs[1].t, outs[2].t, outs[3].t, B, H, N, d,
                             default_scale(d), True, 2, ws.t, wsb)
    _sync_ok()
    assert all(x.intact() for x in outs) and lse.intact() and ws.intact()
