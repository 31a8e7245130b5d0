"""Failure detection on the GPU, without a fault.

Every mbarrier wait in the kernels is bounded: when it runs out it records a
code in the device error word, the CTA stops issuing work, drains what it has
in flight and exits.  fattn_check_wait_timeout (a test hook of
include/fattn_testing.h) runs that same wait routine on a barrier that nothing
ever completes, with a short limit.  The tests check that the timeout is
reported (fattn_device_error returns FATTN_ERR_TIMEOUT; with FATTN_DEBUG set
the entry point itself does), that reading the word clears it, and that the
context still runs the attention kernels correctly afterwards.
"""
import ctypes
import os
import subprocess
import sys

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


def test_device_error_returns_timeout_status():
    lib = fattn.load()
    code = ctypes.c_uint(0)
    assert lib.fattn_device_error(ctypes.byref(code), 1) == 0 and code.value == 0
    fattn.check_wait_timeout()
    assert lib.fattn_device_error(ctypes.byref(code), 0) == 5 and code.value == CHECK_SITE
    assert lib.fattn_device_error(ctypes.byref(code), 1) == 5 and code.value == CHECK_SITE
    assert lib.fattn_device_error(ctypes.byref(code), 1) == 0 and code.value == 0


_DEBUG_CHILD = r"""
import ctypes, sys, torch
sys.path.insert(0, %r)
from online_softmax_08_gb300 import fattn
from online_softmax_08_gb300.inputs import make_inputs, default_scale
lib = fattn.load()
dev = torch.device("cuda:0")
q, k, v = (x.to(dev) for x in make_inputs(1, 1, 256, 64, seed=3))
o, lse = torch.empty_like(q), torch.empty((1, 1, 256), device=dev)
s = torch.cuda.current_stream().cuda_stream
ok = lib.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                   1, 1, 256, 64, default_scale(64), 1, s)
hook = lib.fattn_check_wait_timeout(s)
after = lib.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 1, 256, 64, default_scale(64), 1, s)
code = ctypes.c_uint(0)
cleared = lib.fattn_device_error(ctypes.byref(code), 1)
final = lib.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      1, 1, 256, 64, default_scale(64), 1, s)
print(ok, hook, after, cleared, hex(code.value), final)
"""


def test_debug_mode_returns_timeout_from_the_entry_point():
    """With FATTN_DEBUG=1 every entry point synchronises its stream and reports
    a set error word as FATTN_ERR_TIMEOUT: the hook's own call, and later calls
    until the word is read and cleared."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, FATTN_DEBUG="1")
    out = subprocess.run([sys.executable, "-c", _DEBUG_CHILD % root], env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.split() == ["0", "5", "5", "5", hex(CHECK_SITE), "0"], out.stdout


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
