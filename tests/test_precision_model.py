"""CPU checks of the number-format model that derives tolerances
(tests/bwd_precision_model.py).  Evaluated exactly it must give the
oracle's gradients, its bf16 rounding must be the library routine's, and for
N(0, 1) inputs the bars it derives must sit inside the workloads' 2e-2 bar,
so the bar that only the logit-stress case needs does not widen any other."""
import numpy as np
import pytest
import torch

import bwd_precision_model as bm
import oracle
from online_softmax_08_gb300.inputs import default_scale, make_inputs


def _f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("N,d,causal", [(37, 16, False), (64, 8, True), (130, 32, True)])
def test_exact_model_is_the_oracle(N, d, causal):
    q, k, v, do = (_f64(x) for x in make_inputs(2, 1, N, d, seed=300 + N, with_do=True))
    ref = oracle.attention_bwd(q, k, v, do, 0.3, causal)
    got = bm.backward(q, k, v, do, 0.3, causal, exact=True)
    for a, b in zip(got, ref):
        assert np.abs(a - b).max() <= 1e-10


def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(100000, generator=g) * torch.exp2(torch.randint(-20, 20, (100000,), generator=g).float())
    # exact ties: the low 16 bits equal 0x8000, with both parities of the kept bit
    ties = torch.tensor([0x3F808000, 0x3F818000, 0xBF808000, 0x40008000], dtype=torch.int64)
    ties = torch.from_numpy(ties.numpy().astype(np.uint32).view(np.float32))
    x = torch.cat([x, ties])
    want = x.to(torch.bfloat16).float().numpy()
    assert np.array_equal(bm.bf16_round(x.numpy()), want)


def test_half_ulp_bf16():
    assert bm.half_ulp_bf16(1.0) == 2.0 ** -8
    assert bm.half_ulp_bf16(1.99) == 2.0 ** -8
    assert bm.half_ulp_bf16(9.8) == 2.0 ** -5       # [8, 16): ulp 2^-4
    assert bm.half_ulp_bf16(-0.3) == 2.0 ** -10      # [0.25, 0.5): ulp 2^-9


@pytest.mark.parametrize("N,d,causal", [(300, 64, True), (256, 128, False)])
def test_normal_inputs_fit_the_workload_bars(N, d, causal):
    q, k, v, do = (_f64(x) for x in make_inputs(1, 2, N, d, seed=17 + N, with_do=True))
    s = default_scale(d)
    ref = oracle.attention_bwd(q, k, v, do, s, causal)
    bars, means = bm.derived_bars(q, k, v, do, s, causal, ref, runs=4)
    assert max(bars) <= 2e-2, bars
    assert max(means) <= 2e-3, means
