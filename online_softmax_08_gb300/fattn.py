"""ctypes binding of libfattn (argument marshalling only).

The functions named like the C entry points (``fattn_fwd``, ``fattn_bwd``, ...)
take torch tensors (or raw integer device addresses) and pass their pointers,
sizes and the current CUDA stream straight to the library; every step of the
computation runs in the library's kernels.  ``forward`` and ``backward``
allocate the outputs with torch and then call those entry points.

The library is loaded on first use.  If ``libfattn.so`` is missing the
binding raises: there is no fallback path.
"""
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn.so")

FATTN_OK = 0
STATUS_NAMES = {0: "FATTN_OK", 1: "FATTN_ERR_INVALID_ARG", 2: "FATTN_ERR_UNSUPPORTED",
                3: "FATTN_ERR_CUDA", 4: "FATTN_ERR_WORKSPACE", 5: "FATTN_ERR_TIMEOUT"}

# Every exported symbol of include/fattn.h: name -> (restype, argtypes)
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fattn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fattn_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fattn_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fattn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp,
                       _sz, _vp]),
    "fattn_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i,
                          _vp, _sz, _vp, _vp]),
    "fattn_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f,
                               _i, _vp]),
    "fattn_tile_sizes": (_i, [_i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "fattn_device_error": (_i, [ctypes.POINTER(ctypes.c_uint), _i]),
    "fattn_softmax_rows": (_i, [_vp, _vp, _vp, ctypes.c_longlong, _i, _vp]),
    "fattn_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "fattn_decode_splits": (_i, [_i, _i, _i, _i, _i, _i]),
    "fattn_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fattn_merge_partials": (_i, [_vp, _vp, _i, ctypes.c_longlong, _i, _vp, _vp, _vp]),
    "fattn_fwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fattn_bwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                              _i, _f, _i, _vp, _sz, _vp]),
    "fattn_fwd_bwd_host_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fattn_fwd_bwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f,
                                _i, _i, _vp, _sz, _vp]),
    "fattn_status_string": (ctypes.c_char_p, [_i]),
}

# The test and measurement hooks of include/fattn_testing.h (exported by the
# same library, not part of the attention interface).
TESTING_SIGNATURES = {
    "fattn_check_wait_timeout": (_i, [_vp]),
    "fattn_ex2_throughput": (_i, [ctypes.POINTER(ctypes.c_double), _vp]),
}

_lock = threading.Lock()
_lib = None


class FattnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s returned %s (%d)" % (fn, STATUS_NAMES.get(status, "?"), status))


def load(path=None):
    """Load libfattn.so (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("libfattn.so not found at %s: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in list(SIGNATURES.items()) + list(TESTING_SIGNATURES.items()):
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, status):
    if status != FATTN_OK:
        raise FattnError(name, status)


# ------------------------------------------------------------------ entry points

def fattn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream=None):
    _check("fattn_fwd", load().fattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                         float(scale), int(bool(causal)), _stream(stream)))


def fattn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, tile_counts, stream=None):
    _check("fattn_fwd_ex", load().fattn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H,
                                               N, d, float(scale), int(bool(causal)),
                                               _ptr(tile_counts), _stream(stream)))


def fattn_bwd_workspace_bytes(B, H, N, d):
    return int(load().fattn_bwd_workspace_bytes(B, H, N, d))


def fattn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, workspace,
              workspace_bytes, stream=None):
    _check("fattn_bwd", load().fattn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                         _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                         int(bool(causal)), _ptr(workspace), int(workspace_bytes),
                                         _stream(stream)))


def fattn_bwd_ex(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                 workspace_bytes, phase_events, stream=None):
    """phase_events: None or 4 torch.cuda.Event(enable_timing=True) objects."""
    arr = None
    if phase_events is not None:
        for ev in phase_events:
            if ev.cuda_event == 0:  # torch creates the handle on first record
                ev.record()
        arr = (ctypes.c_void_p * 4)(*[ev.cuda_event for ev in phase_events])
    _check("fattn_bwd_ex", load().fattn_bwd_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H,
        N, d, float(scale), int(bool(causal)), _ptr(workspace), int(workspace_bytes),
        ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None, _stream(stream)))


def fattn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, stream=None):
    """fattn_bwd with the library's built-in workspace (allocates nothing)."""
    _check("fattn_bwd_noalloc", load().fattn_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H,
        N, d, float(scale), int(bool(causal)), _stream(stream)))


def fattn_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, H, max_seqlen, total, d, scale, causal,
                     stream=None):
    _check("fattn_fwd_varlen", load().fattn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), B, H, int(max_seqlen),
        int(total), d, float(scale), int(bool(causal)), _stream(stream)))


def fattn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens, B, H, max_seqlen, total, d,
                     scale, causal, workspace, workspace_bytes, stream=None):
    _check("fattn_bwd_varlen", load().fattn_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(cu_seqlens), B, H, int(max_seqlen), int(total), d, float(scale), int(bool(causal)),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def fattn_fwd_bwd_host_workspace_bytes(B, H, N, d, heads_per_chunk=0):
    return int(load().fattn_fwd_bwd_host_workspace_bytes(B, H, N, d, int(heads_per_chunk)))


def fattn_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, B, H, N, d, scale, causal,
                       heads_per_chunk, workspace, workspace_bytes, stream=None):
    """q, k, v, do, o, lse, dq, dk, dv: HOST tensors (pinned for overlap) or addresses;
    workspace: a device tensor or address."""
    _check("fattn_fwd_bwd_host", load().fattn_fwd_bwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H,
        N, d, float(scale), int(bool(causal)), int(heads_per_chunk), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def fattn_tile_sizes(d, pass_):
    bq, bk = ctypes.c_int(0), ctypes.c_int(0)
    _check("fattn_tile_sizes", load().fattn_tile_sizes(d, pass_, ctypes.byref(bq), ctypes.byref(bk)))
    return bq.value, bk.value


FATTN_ERR_TIMEOUT = 5


def fattn_device_error(clear=True):
    """The device error word (0: no in-kernel wait ran out); the C call returns
    FATTN_ERR_TIMEOUT while the word is set, which is a successful read here."""
    code = ctypes.c_uint(0)
    st = load().fattn_device_error(ctypes.byref(code), int(bool(clear)))
    if st not in (FATTN_OK, FATTN_ERR_TIMEOUT):
        raise FattnError("fattn_device_error", st)
    return code.value


def check_wait_timeout(stream=None):
    """Launch the library's failure-path check (a bounded wait that must give up
    after about 1 ms) on the current stream; read the outcome with
    fattn_device_error()."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check("fattn_check_wait_timeout", load().fattn_check_wait_timeout(s))


def ex2_throughput(stream=None):
    """Measured ex2 evaluations per second of the current device (synchronises)."""
    rate = ctypes.c_double(0.0)
    _check("fattn_ex2_throughput", load().fattn_ex2_throughput(ctypes.byref(rate), _stream(stream)))
    return rate.value


def fattn_status_string(status):
    return load().fattn_status_string(int(status)).decode()


# ------------------------------------------------------------------ allocating wrappers

def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(q.shape)


def forward(q, k, v, scale, causal, tile_counts=None, stream=None):
    """O, LSE of bf16 [B,H,N,d] device tensors q, k, v (contiguous)."""
    B, H, N, d = _shape(q)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if tile_counts is None:
        fattn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)
    else:
        fattn_fwd_ex(q, k, v, o, lse, B, H, N, d, scale, causal, tile_counts, stream)
    return o, lse


def backward(q, k, v, o, lse, do, scale, causal, workspace=None, stream=None):
    """dQ, dK, dV for dL/dO = do.  workspace: None (a torch allocation), a
    device tensor, or "stream" (the library's stream-ordered scratch: the C
    call gets a NULL workspace)."""
    B, H, N, d = _shape(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if isinstance(workspace, str):
        if workspace != "stream":
            raise ValueError(workspace)
        fattn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, None, 0, stream)
        return dq, dk, dv
    nbytes = fattn_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    fattn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, H, N, d, scale, causal, workspace,
              workspace.numel() * workspace.element_size(), stream)
    return dq, dk, dv


def forward_backward_host(q, k, v, do, scale, causal, heads_per_chunk=0, workspace=None,
                          device=None, stream=None):
    """Forward and backward of HOST bf16 tensors [B,H,N,d] through the device:
    returns HOST (o, lse, dq, dk, dv), page-locked.  The call is asynchronous on
    the stream; synchronise before reading the results."""
    B, H, N, d = _shape(q)
    device = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(device):
        if stream is None:
            stream = torch.cuda.current_stream(device)
        nbytes = fattn_fwd_bwd_host_workspace_bytes(B, H, N, d, heads_per_chunk)
        own = workspace is None
        if own:
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
        o, dq, dk, dv = (torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4))
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        fattn_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, B, H, N, d, scale, causal,
                           heads_per_chunk, workspace, workspace.numel() * workspace.element_size(),
                           stream)
        if own and isinstance(stream, torch.cuda.Stream):
            # the workspace is in use until `stream` passes the call: keep the
            # allocator from handing it out before then
            workspace.record_stream(stream)
    return o, lse, dq, dk, dv


def forward_varlen(q, k, v, cu_seqlens, max_seqlen, scale, causal, stream=None):
    """O, LSE of packed bf16 [H, total, d] device tensors; cu_seqlens is a device
    int32 tensor of B + 1 offsets (its last entry, total, is q.shape[1])."""
    H, T, d = q.shape
    B = cu_seqlens.numel() - 1
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    fattn_fwd_varlen(q, k, v, o, lse, cu_seqlens, B, H, max_seqlen, T, d, scale, causal, stream)
    return o, lse


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen, scale, causal, workspace=None,
                    stream=None):
    """dQ, dK, dV of forward_varlen for dL/dO = do."""
    H, T, d = q.shape
    B = cu_seqlens.numel() - 1
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(max(fattn_bwd_workspace_bytes(1, H, max(T, 1), d), 1),
                                dtype=torch.uint8, device=q.device)
    fattn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, cu_seqlens, B, H, max_seqlen, T, d, scale,
                     causal, workspace, workspace.numel() * workspace.element_size(), stream)
    return dq, dk, dv


def decode(q, k, v, scale, causal, n_splits=0, workspace=None, stream=None):
    """O, LSE of few queries q [B,H,Nq,d] against k, v [B,H,Nkv,d] (the queries
    are the last Nq positions) by split-KV plus merge."""
    B, H, Nq, d = _shape(q)
    Nkv = k.shape[2]
    lib = load()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    nbytes = int(lib.fattn_decode_workspace_bytes(B, H, Nq, Nkv, d, n_splits))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check("fattn_decode", lib.fattn_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nkv, d, float(scale),
        int(bool(causal)), int(n_splits), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def merge_partials(o_part, lse_part, stream=None):
    """Merge fp32 partials o_part [S, rows, d], lse_part [S, rows] -> bf16 o [rows, d], lse."""
    S, rows, d = o_part.shape
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=o_part.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_part.device)
    _check("fattn_merge_partials", load().fattn_merge_partials(
        _ptr(o_part), _ptr(lse_part), S, rows, d, _ptr(o), _ptr(lse), _stream(stream)))
    return o, lse


def softmax_rows(x, with_lse=False, out=None, stream=None):
    """Row-wise softmax of a contiguous fp32 [rows, cols] device tensor."""
    rows, cols = x.shape
    y = torch.empty_like(x) if out is None else out
    lse = torch.empty((rows,), dtype=torch.float32, device=x.device) if with_lse else None
    _check("fattn_softmax_rows", load().fattn_softmax_rows(_ptr(x), _ptr(y), _ptr(lse), rows, cols,
                                                           _stream(stream)))
    return (y, lse) if with_lse else y
