"""ctypes binding of libfattn_host (argument marshalling only).

libfattn_host is the flash-style attention forward pass on the host CPU cores
(fp32, OpenMP), a separate library from the GPU's libfattn: nothing here is
called by the GPU entry points and nothing here calls them.  The functions
take numpy arrays (or CPU torch tensors), check shapes and dtypes, and pass
pointers and sizes straight to the library.  If ``libfattn_host.so`` is
missing the binding raises.
"""
import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn_host.so")

STATUS_NAMES = {0: "FATTN_HOST_OK", 1: "FATTN_HOST_ERR_INVALID_ARG",
                2: "FATTN_HOST_ERR_UNSUPPORTED", 6: "FATTN_HOST_ERR_NO_MEMORY"}
MAX_D = 256

_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
# Every exported symbol of include/fattn_host.h: name -> (restype, argtypes)
SIGNATURES = {
    "fattn_host_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i]),
    "fattn_host_max_threads": (_i, []),
    "fattn_host_fma_peak_gflops": (ctypes.c_double, [_i, ctypes.c_double]),
    "fattn_host_exp2": (None, [_vp, _vp, ctypes.c_longlong]),
}

_lock = threading.Lock()
_lib = None


class FattnHostError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s returned %s (%d)" % (fn, STATUS_NAMES.get(status, "?"), status))


def load(path=None):
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise FileNotFoundError("%s is not built (run the package build)" % p)
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
        return _lib


def _array(x, name):
    if hasattr(x, "numpy"):  # a CPU torch tensor
        x = x.detach().numpy()
    if not isinstance(x, np.ndarray) or x.dtype != np.float32 or not x.flags.c_contiguous:
        raise TypeError("%s must be a C-contiguous float32 array" % name)
    return x


def fattn_host_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, n_threads=0):
    st = load().fattn_host_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                               lse.ctypes.data, B, H, N, d, scale, int(bool(causal)),
                               int(n_threads))
    if st != 0:
        raise FattnHostError("fattn_host_fwd", st)


def forward(q, k, v, scale, causal, n_threads=0):
    """O [B,H,N,d] and LSE [B,H,N] (float32 numpy arrays) of fp32 q, k, v [B,H,N,d]."""
    q, k, v = _array(q, "q"), _array(k, "k"), _array(v, "v")
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float32)
    fattn_host_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, n_threads)
    return o, lse


def max_threads():
    return load().fattn_host_max_threads()


def fma_peak_gflops(n_threads=0, seconds=0.3):
    return load().fattn_host_fma_peak_gflops(int(n_threads), float(seconds))


def exp2(t):
    t = np.ascontiguousarray(t, dtype=np.float32)
    y = np.empty_like(t)
    load().fattn_host_exp2(t.ctypes.data, y.ctypes.data, t.size)
    return y
