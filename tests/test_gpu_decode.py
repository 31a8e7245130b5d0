"""Split-KV decoding and the block-state merge against the fp64 oracle.

fattn_decode: few queries (the last Nq positions) against many keys; the key
tiles are cut into ranges, one per CTA, and merged.  Cases cover one query,
sixteen, more than one 128-row subtile, ragged key counts, both head sizes,
forced split counts from one range to one range per tile, and Nq == Nkv (the
dense forward's problem).  fattn_merge_partials is checked on its own against
the oracle's block-wise merge, including rows whose ranges saw no key.
Bar: O max-abs <= 2e-2 and mean-abs <= 2e-3, LSE <= 1e-3 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _qkv(B, H, Nq, Nkv, d, seed):
    q, k, v = make_inputs(B, H, Nkv, d, seed)
    return q[:, :, Nkv - Nq:].contiguous(), k, v


CASES = [
    # B, H, Nq, Nkv, d, causal, n_splits
    (2, 4, 1, 5000, 128, True, 0),
    (2, 4, 1, 5000, 128, False, 0),
    (1, 8, 16, 3000, 64, True, 0),
    (1, 2, 200, 1000, 128, True, 0),
    (1, 2, 7, 1300, 128, True, 1),
    (1, 2, 7, 1300, 128, True, 3),
    (1, 2, 7, 1300, 128, False, 1000),
    (1, 1, 384, 384, 128, True, 0),
]


@pytest.mark.parametrize("B,H,Nq,Nkv,d,causal,n_splits", CASES)
def test_decode_matches_oracle(B, H, Nq, Nkv, d, causal, n_splits):
    q, k, v = _qkv(B, H, Nq, Nkv, d, seed=700 + Nq + Nkv + d)
    dev = torch.device("cuda:0")
    scale = default_scale(d)
    o, lse = fattn.decode(q.to(dev), k.to(dev), v.to(dev), scale, causal, n_splits)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    o_ref, lse_ref = oracle.attention_fwd_decode(_f64(q), _f64(k), _f64(v), scale, causal)
    err = np.abs(_f64(o) - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(_f64(lse) - lse_ref).max() <= LSE_MAX


def _expected_splits(units, Nq, Nkv, n_splits, n_sm):
    """The documented rule: a request is capped at one range per 128-key tile;
    0 asks for about ten waves of CTAs over the device's SMs with at least four
    tiles per range; empty ranges are dropped."""
    n_tiles = -(-Nkv // 128)
    want = n_splits
    if want <= 0:
        ctas = units * -(-Nq // 256)
        want = min(-(-10 * n_sm // ctas), n_tiles // 4)
    want = max(1, min(want, n_tiles))
    tps = -(-n_tiles // want)
    return -(-n_tiles // tps)


def test_split_counts():
    lib = fattn.load()
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    for args in [(1, 1, 1, 1300, 1000), (1, 1, 1, 1300, 3), (4, 32, 1, 32768, 0),
                 (1, 1, 1, 1300, 0), (2, 8, 300, 70000, 0), (16, 64, 1, 4096, 0)]:
        B, H, Nq, Nkv, n = args
        assert lib.fattn_decode_splits(B, H, Nq, Nkv, 128, n) == \
            _expected_splits(B * H, Nq, Nkv, n, n_sm), args
    assert lib.fattn_decode_splits(1, 1, 1, 1300, 128, 1000) == 11  # one range per tile
    assert lib.fattn_decode_splits(1, 1, 1, 1300, 128, 3) == 3
    assert lib.fattn_decode_splits(1, 1, 2, 1, 128, 0) == 0  # Nq > Nkv is invalid


@pytest.mark.parametrize("S,rows,d", [(1, 5, 128), (4, 300, 64), (37, 64, 128)])
def test_merge_partials_matches_oracle(S, rows, d):
    g = torch.Generator().manual_seed(S * 1000 + rows + d)
    o_part = torch.randn((S, rows, d), generator=g, dtype=torch.float32)
    lse_part = torch.randn((S, rows), generator=g, dtype=torch.float32) * 4.0
    if S > 1:
        lse_part[1, ::3] = -float("inf")   # some ranges saw no key for some rows
        o_part[1, ::3] = 0.0
    lse_part[:, 1] = -float("inf")         # a row that saw no key at all
    o_part[:, 1] = 0.0
    dev = torch.device("cuda:0")
    o, lse = fattn.merge_partials(o_part.to(dev), lse_part.to(dev))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge_partials(o_part.double().numpy(), lse_part.double().numpy())
    assert np.abs(_f64(o) - o_ref).max() <= 2e-2
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(_f64(lse)), finite)
    assert np.abs(_f64(lse)[finite] - lse_ref[finite]).max() <= 1e-5
    assert np.all(_f64(o)[1] == 0.0)


def test_decode_bench_workload_full():
    """The benchmark's decoding workload (B4 H32, one query against 32768
    keys, d128, automatic key ranges), every output row against the oracle."""
    from online_softmax_08_gb300.inputs import DECODE_WORKLOADS
    w = DECODE_WORKLOADS["decode_b4h32_nq1_nkv32768_d128"]
    B, H, Nq, Nkv, d = w["B"], w["H"], w["Nq"], w["Nkv"], w["d"]
    q, k, v = make_inputs(B, H, Nkv, d, w["seed"])
    q = q[:, :, Nkv - Nq:].contiguous()
    dev = torch.device("cuda:0")
    scale = default_scale(d)
    o, lse = fattn.decode(q.to(dev), k.to(dev), v.to(dev), scale, w["causal"])
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    o_ref, lse_ref = oracle.attention_fwd_decode(_f64(q), _f64(k), _f64(v), scale, w["causal"])
    err = np.abs(_f64(o) - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    assert np.abs(_f64(lse) - lse_ref).max() <= LSE_MAX
