"""The C-ABI libraries load and export every entry point their headers declare
(include/fattn.h and the test hooks of include/fattn_testing.h: libfattn;
include/fattn_host.h: libfattn_host); argument checks that fail before any
device work run on the CPU."""
import os
import re

import pytest

from online_softmax_08_gb300 import build as fbuild
from online_softmax_08_gb300 import fattn, fattn_host

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fattn.load()


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    return set(re.findall(r"^\s*(?:int|size_t|double|void|const char\*)\s+(fattn_\w+)\s*\(",
                          src, flags=re.M))


def test_headers_are_the_two_libraries():
    assert sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")) == \
        ["fattn.h", "fattn_host.h", "fattn_testing.h"]


def test_every_declared_symbol_is_exported_and_bound(lib):
    declared = _declared("fattn.h")
    assert {"fattn_fwd", "fattn_bwd", "fattn_bwd_workspace_bytes"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
        assert name in fattn.SIGNATURES, name
    assert set(fattn.SIGNATURES) == declared


def test_test_hooks_are_declared_apart(lib):
    hooks = _declared("fattn_testing.h")
    assert hooks == {"fattn_check_wait_timeout", "fattn_ex2_throughput"}
    assert not hooks & _declared("fattn.h")
    for name in hooks:
        assert hasattr(lib, name), name
    assert set(fattn.TESTING_SIGNATURES) == hooks


def test_every_host_symbol_is_exported_and_bound(lib):
    host = fattn_host.load()
    declared = _declared("fattn_host.h")
    assert {"fattn_host_fwd", "fattn_host_fma_peak_gflops"} <= declared
    for name in declared:
        assert hasattr(host, name), name
    assert set(fattn_host.SIGNATURES) == declared


def test_status_strings(lib):
    assert fattn.fattn_status_string(0) == "ok"
    assert "workspace" in fattn.fattn_status_string(4)


def test_tile_sizes(lib):
    assert fattn.fattn_tile_sizes(128, 0) == (128, 128)
    assert fattn.fattn_tile_sizes(64, 0) == (128, 128)
    assert fattn.fattn_tile_sizes(128, 1) == (128, 128)
    assert fattn.fattn_tile_sizes(64, 1) == (128, 128)
    with pytest.raises(fattn.FattnError):
        fattn.fattn_tile_sizes(96, 0)


def test_workspace_bytes(lib):
    n = fattn.fattn_bwd_workspace_bytes(2, 3, 100, 64)
    rows = 2 * 3 * 100
    assert n >= rows * 64 * 4 + rows * 4 and n % 256 == 0
    assert fattn.fattn_bwd_workspace_bytes(1, 1, 1, 96) == 0


def test_argument_checks_before_any_device_call(lib):
    # every call here fails validation, which happens before the library
    # touches the CUDA runtime, so no GPU is needed
    a = 1 << 20  # a 16-byte-aligned address that is never dereferenced
    assert lib.fattn_fwd(None, a, a, a, a, 1, 1, 128, 128, 0.1, 0, None) == 1
    assert lib.fattn_fwd(a + 8, a, a, a, a, 1, 1, 128, 128, 0.1, 0, None) == 1
    assert lib.fattn_fwd(a, a, a, a, a, 1, 1, 128, 80, 0.1, 0, None) == 2
    assert lib.fattn_fwd(a, a, a, a, a, 0, 1, 128, 128, 0.1, 0, None) == 1
    assert lib.fattn_fwd(a, a, a, a, a, 1, 1, 128, 128, 0.0, 0, None) == 1
    assert lib.fattn_fwd(a, a, a, a, a, 1 << 16, 1 << 16, 1, 64, 0.1, 0, None) == 1
    assert lib.fattn_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 128, 0.1, 1, a + 16, 1 << 30,
                         None) == 4
    assert lib.fattn_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 128, 0.1, 1, a, 16, None) == 4


def test_ex2_probe_checks_its_pointer_first(lib):
    assert lib.fattn_ex2_throughput(None, None) == 1


def test_host_staged_argument_checks_before_any_device_call(lib):
    a = 1 << 20
    ws = 1 << 24  # 256-byte aligned, never dereferenced
    args = lambda **kw: [kw.get(n, a) for n in ("q", "k", "v", "do", "o", "lse", "dq", "dk", "dv")]
    call = lambda ptrs, B=1, H=4, N=256, d=64, scale=0.1, hpc=2, w=ws, wb=1 << 40: \
        lib.fattn_fwd_bwd_host(*ptrs, B, H, N, d, scale, 1, hpc, w, wb, None)
    assert call(args(q=None)) == 1
    assert call(args(lse=None)) == 1
    assert call(args(), d=80) == 2
    assert call(args(), B=0) == 1
    assert call(args(), scale=float("inf")) == 1
    assert call(args(), hpc=-1) == 1
    assert call(args(), w=None) == 4
    assert call(args(), w=ws + 128) == 4
    need = fattn.fattn_fwd_bwd_host_workspace_bytes(1, 4, 256, 64, 2)
    assert call(args(), wb=need - 1) == 4
    # three slots, each with 8 bf16 tiles, LSE and the backward's workspace of 2 heads
    rows = 2 * 256
    assert need == 3 * (8 * rows * 64 * 2 + rows * 4 + fattn.fattn_bwd_workspace_bytes(1, 2, 256, 64))
    assert fattn.fattn_fwd_bwd_host_workspace_bytes(1, 4, 256, 96, 2) == 0
    # a chunk larger than B*H is clipped to B*H
    assert fattn.fattn_fwd_bwd_host_workspace_bytes(1, 4, 256, 64, 9) == \
        fattn.fattn_fwd_bwd_host_workspace_bytes(1, 4, 256, 64, 4)


def test_null_workspace_passes_validation(lib):
    """A NULL workspace asks for stream-ordered scratch: the arguments pass, and
    the call proceeds to the device (without one: FATTN_ERR_CUDA)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    a = 1 << 20
    assert lib.fattn_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 128, 0.1, 1, None, 0, None) == 3
    # validation still comes first
    assert lib.fattn_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 96, 0.1, 1, None, 0, None) == 2


def test_noalloc_checks_arguments_like_fattn_bwd(lib):
    a = 1 << 20
    # B = 0 with an unsupported d: the size check comes first, as in fattn_bwd
    for fn in ("fattn_bwd_noalloc",):
        f = getattr(lib, fn)
        assert f(a, a, a, a, a, a, a, a, a, 0, 1, 128, 32, 0.1, 1, None) == 1
        # a bad scale on a problem beyond the built-in scratch: INVALID_ARG, not WORKSPACE
        assert f(a, a, a, a, a, a, a, a, a, 1, 8, 16384, 128, float("nan"), 1, None) == 1
        assert f(a, a, a, a, a, a, a, a, a, 1, 8, 16384, 128, -1.0, 1, None) == 1
        assert f(a, a, a, a, a, a, a, a, a, 1, 1, 128, 96, 0.1, 1, None) == 2
        assert f(a, a, a, a, a, a, a, a, a, 1, 8, 16384, 128, 0.1, 1, None) == 4
    big = (1 << 16, 1 << 16, 1)
    assert lib.fattn_bwd_noalloc(a, a, a, a, a, a, a, a, a, *big, 64, 0.1, 0, None) == 1
    assert lib.fattn_bwd(a, a, a, a, a, a, a, a, a, *big, 64, 0.1, 0, a, 1 << 40, None) == 1
