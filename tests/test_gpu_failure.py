"""Failure detection on the GPU, without a fault.

Every mbarrier wait in the kernels is bounded: when it runs out it records a
code in the device error word, the CTA stops issuing work, drains what it has
in flight and exits.  fattn_check_wait_timeout runs that same wait routine on
a barrier that nothing ever completes, with a short limit.  The tests check
that the timeout is reported, that reading the word clears it, and that the
context still runs the attention kernels correctly afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import default_scale, make_inputs

pytestmark = pytest.mark.gpu

CHECK_SITE = 0x301  # ERR_SITE_CHECK | 1


def test_bounded_wait_reports_timeout_and_context_survives():
    assert fattn.fattn_device_error(clear=True) == 0
    fattn.check_wait_timeout()  # gives up after about 1 ms
    torch.cuda.synchronize()
    assert fattn.fattn_device_error(clear=True) == CHECK_SITE
    assert fattn.fattn_device_error(clear=True) == 0  # reading with clear resets it

    # the context is still usable: a forward pass right after matches the oracle
    q, k, v = make_inputs(1, 2, 300, 128, seed=515)
    dev = torch.device("cuda:0")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    scale = default_scale(128)
    o, lse = fattn.forward(qd, kd, vd, scale, True)
    torch.cuda.synchronize()
    assert fattn.fattn_device_error() == 0
    f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
    o_ref, lse_ref = oracle.attention_fwd(f64(q), f64(k), f64(v), scale, True)
    assert np.abs(f64(o) - o_ref).max() <= 2e-2
    assert np.abs(f64(lse) - lse_ref).max() <= 1e-3


def test_first_failure_wins():
    fattn.check_wait_timeout()
    fattn.check_wait_timeout()
    torch.cuda.synchronize()
    assert fattn.fattn_device_error(clear=False) == CHECK_SITE
    assert fattn.fattn_device_error(clear=True) == CHECK_SITE
    assert fattn.fattn_device_error() == 0


def test_ex2_throughput_probe_is_plausible():
    """The measured ex2 rate (the forward pass's second ceiling) lies between
    1e12/s and 2e13/s on a GB300 (16 per clock per SM x 152 SMs x about 2 GHz
    is about 5e12/s)."""
    rate = fattn.ex2_throughput()
    assert 1e12 < rate < 2e13, rate
