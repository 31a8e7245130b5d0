"""Variable-length batches: libfattn's packed-sequence entry points against the
fp64 oracle applied to each sequence.

Layout [H, T, d] with sequence b at rows [cu[b], cu[b+1]).  Lengths are chosen
to cross tile boundaries (1, 127, 128, 129, ...), to leave a ragged last tile
whose rows belong to the next sequence, and to include an empty sequence.
Bar: the dense bar (O, dQ, dK, dV max-abs <= 2e-2, mean-abs <= 2e-3; LSE
<= 1e-3), element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_varlen_inputs

pytestmark = pytest.mark.gpu

MAX, MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3

CASES = [
    # (lengths, H, d, causal)
    ([1, 127, 128, 129, 300], 2, 128, True),
    ([1, 127, 128, 129, 300], 2, 128, False),
    ([777, 0, 64, 1000], 2, 64, True),
    ([256, 256, 256], 3, 64, False),
    ([5, 1300, 3], 1, 128, True),
    # equal lengths among others: CTAs take sequences longest first, ties by index
    ([300, 200, 300, 128, 0, 300, 256, 700], 2, 128, True),
    # more sequences than the longest-first ordering handles: index order
    ([(37 * i) % 301 for i in range(70)], 1, 64, True),
]


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _close(got, want):
    err = np.abs(got - want)
    assert np.isfinite(got).all()
    assert err.max() <= MAX, err.max()
    assert err.mean() <= MEAN, err.mean()


@pytest.mark.parametrize("lengths,H,d,causal", CASES)
def test_varlen_forward_and_backward_match_oracle(lengths, H, d, causal):
    q, k, v, do, cu = make_varlen_inputs(lengths, H, d, seed=808 + sum(lengths) + d, with_do=True)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod, cud = (x.to(dev) for x in (q, k, v, do, cu))
    scale = default_scale(d)
    o, lse = fattn.forward_varlen(qd, kd, vd, cud, max(lengths), scale, causal)
    dq, dk, dv = fattn.backward_varlen(qd, kd, vd, o, lse, dod, cud, max(lengths), scale, causal)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    o_ref, lse_ref = oracle.attention_fwd_varlen(_f64(q), _f64(k), _f64(v), cu.numpy(), scale, causal)
    _close(_f64(o), o_ref)
    assert np.abs(_f64(lse) - lse_ref).max() <= LSE_MAX
    g_ref = oracle.attention_bwd_varlen(_f64(q), _f64(k), _f64(v), _f64(do), cu.numpy(), scale,
                                        causal)
    for got, want in zip((dq, dk, dv), g_ref):
        _close(_f64(got), want)


@pytest.mark.parametrize("d", [64, 128])
def test_repeated_varlen_backward_calls(d):
    """Repeated varlen backward calls agree: dK and dV bit for bit, dQ within one bf16
    step.  Lengths off multiples of 32 and 128 leave the dQ boxes of a sequence's
    last query block reaching into the next sequence's rows (adding exact zeros)
    while that sequence's own CTAs add into them."""
    lengths = [777, 95, 1000, 33, 513, 260]
    q, k, v, do, cu = make_varlen_inputs(lengths, 3, d, seed=1944 + d, with_do=True)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod, cud = (x.to(dev) for x in (q, k, v, do, cu))
    scale = default_scale(d)
    for causal in (False, True):
        o, lse = fattn.forward_varlen(qd, kd, vd, cud, max(lengths), scale, causal)
        dq0, dk0, dv0 = fattn.backward_varlen(qd, kd, vd, o, lse, dod, cud, max(lengths), scale,
                                              causal)
        for _ in range(15):
            dq, dk, dv = fattn.backward_varlen(qd, kd, vd, o, lse, dod, cud, max(lengths), scale,
                                               causal)
            assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
            a, b = dq.float(), dq0.float()
            assert bool(((a - b).abs() <= torch.maximum(a.abs(), b.abs()) * 2.0**-7 + 1e-5).all())
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0


def test_varlen_d64_grid_of_two_subtile_ctas():
    """The d = 64 varlen forward on a grid large enough (from the device's SM
    count) for two 128-row subtiles per CTA, forward and backward against the
    oracle on every sequence."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    H, d = 8, 64
    n_seq = -(-(6 * n_sm + 1) // (H * 8))  # 8 blocks of 256 rows for the longest sequence
    lengths = [2048] + [(97 * i) % 1500 + 1 for i in range(1, n_seq)]
    assert n_seq * H * 8 > 6 * n_sm
    test_varlen_forward_and_backward_match_oracle(lengths, H, d, True)


def test_varlen_with_equal_lengths_equals_the_dense_kernels():
    """The packed path on B equal-length sequences gives the dense path's bits
    for O and LSE (the same tiles, masks and order) and the same gradients to
    within the order of the fp32 dQ reductions."""
    B, H, N, d = 3, 2, 640, 128
    q, k, v, do, cu = make_varlen_inputs([N] * B, H, d, seed=901, with_do=True)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod, cud = (x.to(dev) for x in (q, k, v, do, cu))
    scale = default_scale(d)
    o, lse = fattn.forward_varlen(qd, kd, vd, cud, N, scale, True)
    dq, dk, dv = fattn.backward_varlen(qd, kd, vd, o, lse, dod, cud, N, scale, True)
    dense = lambda x: x.reshape(H, B, N, d).transpose(0, 1).contiguous()
    o2, lse2 = fattn.forward(dense(qd), dense(kd), dense(vd), scale, True)
    g2 = fattn.backward(dense(qd), dense(kd), dense(vd), o2, lse2, dense(dod), scale, True)
    torch.cuda.synchronize()
    assert torch.equal(dense(o), o2)
    assert torch.equal(lse.reshape(H, B, N).transpose(0, 1), lse2)
    assert torch.equal(dense(dk), g2[1]) and torch.equal(dense(dv), g2[2])
    assert (dense(dq).float() - g2[0].float()).abs().max().item() <= 2e-3


def test_bad_offsets_are_reported_not_used():
    """A decreasing offset (sequence 1 below) or a sequence longer than
    max_seqlen is skipped on the device and reported through the error word;
    nothing is written for it."""
    dev = torch.device("cuda:0")
    H, d, T = 1, 128, 300
    q, k, v, _ = make_varlen_inputs([T], H, d, seed=902)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    assert fattn.fattn_device_error() == 0
    cu = torch.tensor([0, 200, 100, 300], dtype=torch.int32, device=dev)
    o = torch.full_like(qd, 7.0)
    lse = torch.full((H, T), 7.0, device=dev)
    fattn.fattn_fwd_varlen(qd, kd, vd, o, lse, cu, 3, H, 200, T, d, default_scale(d), True)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0x140
    # sequences 0 ([0, 200)) and 2 ([100, 300)) were computed; sequence 1 was not
    assert torch.isfinite(o).all()
    cu = torch.tensor([0, 300], dtype=torch.int32, device=dev)
    fattn.fattn_fwd_varlen(qd, kd, vd, o, lse, cu, 1, H, 200, T, d, default_scale(d), True)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0x140
    assert fattn.fattn_device_error() == 0


def test_varlen_bench_workload_sampled():
    """The benchmark's packed workload (16 sequences, lengths uniform in
    [512, 8192], H16 d128 causal), run as the benchmark runs it: forward rows
    sampled in every sequence for two heads, each row computed by the oracle
    one by one; the backward of one head checked in full on the two shortest
    sequences."""
    from online_softmax_08_gb300.inputs import VARLEN_WORKLOADS, varlen_lengths
    w = VARLEN_WORKLOADS["varlen_b16h16_len512to8192_d128_causal"]
    H, d = w["H"], w["d"]
    lens = varlen_lengths(w["B"], w["lo"], w["hi"], w["seed"])
    q, k, v, do, cu = make_varlen_inputs(lens, H, d, w["seed"], with_do=True)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod, cud = (x.to(dev) for x in (q, k, v, do, cu))
    scale = default_scale(d)
    o, lse = fattn.forward_varlen(qd, kd, vd, cud, max(lens), scale, True)
    dq, dk, dv = fattn.backward_varlen(qd, kd, vd, o, lse, dod, cud, max(lens), scale, True)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    of, lf = _f64(o), _f64(lse)
    rng = np.random.default_rng(w["seed"])
    cu_np = cu.numpy()
    for b in range(len(lens)):
        a, e = int(cu_np[b]), int(cu_np[b + 1])
        rows = np.unique(np.concatenate([[0, e - a - 1], rng.integers(0, e - a, 6)]))
        sl = lambda x: _f64(x[:, a:e])[None]
        heads = np.array([0, H - 1])
        bh = np.repeat(heads, len(rows))
        rr = np.tile(rows, len(heads))
        o_ref, lse_ref = oracle.attention_fwd_rows(sl(q), sl(k), sl(v), scale, True, bh, rr)
        got = of[bh, a + rr]
        assert np.abs(got - o_ref).max() <= MAX
        assert np.abs(lf[bh, a + rr] - lse_ref).max() <= LSE_MAX
    for b in np.argsort(lens)[:2]:
        a, e = int(cu_np[b]), int(cu_np[b + 1])
        sl = lambda x: _f64(x[:, a:e])[None]
        g_ref = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), scale, True, heads=[3])
        for got, want in zip((dq, dk, dv), g_ref):
            _close(_f64(got[3:4, a:e]), want)
