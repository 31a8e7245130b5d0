"""fp64 CPU oracle for scaled dot-product attention.  TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  It is independent of the CUDA path:
the two share no code, and nothing here imports ``online_softmax_08_gb300``.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP loops); this module
compiles it on demand with gcc and marshals numpy arrays through ctypes.

  attention_fwd       -- S = scale Q K^T, three-pass safe softmax, O = P V, LSE
  attention_fwd_rows  -- the same definition for sampled (head, query row) pairs
  attention_bwd       -- the textbook backward (dQ, dK, dV) of that definition
  tile_counts         -- brute-force full / masked / skipped tile classification
  attention_fwd_varlen, attention_bwd_varlen
                      -- packed variable-length batches: each sequence is its own
                         attention problem (the definition applied per sequence)
  attention_fwd_decode
                      -- few queries at the end of a long sequence (numpy, fp64)
  merge_partials      -- block states (o_s, lse_s) over disjoint key ranges
                         merged by the block-wise update (numpy, fp64)
  softmax_rows        -- row-wise safe softmax and its log-sum-exp (numpy, fp64)

Inputs are numpy float64 arrays of shape [B, H, N, d] (contiguous).
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_int64)
        i64, c_int, c_double = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, c_double, c_int, c_int]
        lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, i64, i64, i64, c_double, c_int, lp, lp,
                                             i64, dp, dp, c_int]
        lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, c_double, c_int, lp, i64,
                                        dp, dp, dp, c_int]
        lib.oracle_tile_counts.argtypes = [i64, c_int, i64, i64, lp]
        lib.oracle_max_threads.argtypes = []
        for f in (lib.oracle_attn_fwd, lib.oracle_attn_fwd_rows, lib.oracle_attn_bwd,
                  lib.oracle_tile_counts, lib.oracle_max_threads):
            f.restype = c_int
        _lib = lib
        return lib


def _f64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _i64(a):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (what, rc))


def max_threads():
    return _load().oracle_max_threads()


def attention_fwd(q, k, v, scale, causal, nthreads=0):
    """O [B,H,N,d] and LSE [B,H,N] (natural log) of softmax(scale Q K^T) V."""
    lib = _load()
    B, H, N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    o, op = _f64(np.empty((B, H, N, d)))
    lse, lp_ = _f64(np.empty((B, H, N)))
    _check(lib.oracle_attn_fwd(qp, kp, vp, op, lp_, B * H, N, d, float(scale), int(bool(causal)),
                               int(nthreads)), "fwd")
    return o, lse


def attention_fwd_rows(q, k, v, scale, causal, bh_idx, row_idx, nthreads=0):
    """Output rows o [count, d] and lse [count] for the sampled (b*H+h, row) pairs."""
    lib = _load()
    B, H, N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    bh, bhp = _i64(bh_idx)
    rows, rp = _i64(row_idx)
    if bh.shape != rows.shape:
        raise ValueError("bh_idx and row_idx differ in length")
    o, op = _f64(np.empty((len(rows), d)))
    lse, lp_ = _f64(np.empty((len(rows),)))
    _check(lib.oracle_attn_fwd_rows(qp, kp, vp, B * H, N, d, float(scale), int(bool(causal)), bhp,
                                    rp, len(rows), op, lp_, int(nthreads)), "fwd_rows")
    return o, lse


def attention_bwd(q, k, v, do, scale, causal, heads=None, nthreads=0):
    """dQ, dK, dV of sum(O * dO).  With ``heads`` (flat b*H+h indices) only those
    heads are computed and the outputs are [len(heads), N, d]; otherwise
    [B, H, N, d]."""
    lib = _load()
    B, H, N, d = q.shape
    q, qp = _f64(q)
    k, kp = _f64(k)
    v, vp = _f64(v)
    do, dop = _f64(do)
    if heads is None:
        nh, hp, shape = B * H, None, (B, H, N, d)
    else:
        hs, hp = _i64(heads)
        nh, shape = len(hs), (len(hs), N, d)
    dq, dqp = _f64(np.empty(shape))
    dk, dkp = _f64(np.empty(shape))
    dv, dvp = _f64(np.empty(shape))
    _check(lib.oracle_attn_bwd(qp, kp, vp, dop, B * H, N, d, float(scale), int(bool(causal)), hp, nh,
                               dqp, dkp, dvp, int(nthreads)), "bwd")
    return dq, dk, dv


def tile_counts(N, causal, block_q, block_k):
    """(full, masked, skipped) tiles of one head's grid."""
    lib = _load()
    out, op = _i64(np.zeros(3))
    _check(lib.oracle_tile_counts(int(N), int(bool(causal)), int(block_q), int(block_k), op), "tiles")
    return tuple(int(x) for x in out)


def _sequences(cu_seqlens):
    cu = [int(x) for x in cu_seqlens]
    if cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must start at 0 and not decrease")
    return list(zip(cu[:-1], cu[1:]))


def attention_fwd_varlen(q, k, v, cu_seqlens, scale, causal, nthreads=0):
    """O [H,T,d] and LSE [H,T] of a packed batch: q, k, v are [H, T, d] with
    sequence b at rows [cu[b], cu[b+1]).  Each sequence is an independent
    attention problem; the definition (attention_fwd) is applied to each slice.
    Rows that belong to no sequence (none, when cu[-1] == T) stay NaN."""
    H, T, d = q.shape
    o = np.full((H, T, d), np.nan)
    lse = np.full((H, T), np.nan)
    for a, b in _sequences(cu_seqlens):
        if b == a:
            continue
        sl = lambda x: np.ascontiguousarray(x[:, a:b][None])
        os_, ls_ = attention_fwd(sl(q), sl(k), sl(v), scale, causal, nthreads)
        o[:, a:b], lse[:, a:b] = os_[0], ls_[0]
    return o, lse


def attention_bwd_varlen(q, k, v, do, cu_seqlens, scale, causal, nthreads=0):
    """dQ, dK, dV [H,T,d] of a packed batch (see attention_fwd_varlen)."""
    H, T, d = q.shape
    dq, dk, dv = (np.full((H, T, d), np.nan) for _ in range(3))
    for a, b in _sequences(cu_seqlens):
        if b == a:
            continue
        sl = lambda x: np.ascontiguousarray(x[:, a:b][None])
        g = attention_bwd(sl(q), sl(k), sl(v), sl(do), scale, causal, None, nthreads)
        dq[:, a:b], dk[:, a:b], dv[:, a:b] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


def attention_fwd_decode(q, k, v, scale, causal):
    """O [B,H,Nq,d], LSE [B,H,Nq] for queries that are the LAST Nq positions of a
    sequence of Nkv keys: query i sits at position Nkv - Nq + i and, with
    causal, sees keys j <= Nkv - Nq + i.  The definition written out in numpy
    fp64: S = scale Q K^T, the mask, the three-pass safe softmax of page
    "tm_flash_attention_math" ("Safe softmax"), O = P V, LSE = m + ln l."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, H, Nq, d = q.shape
    Nkv = k.shape[2]
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        pos = np.arange(Nq)[:, None] + (Nkv - Nq)
        s = np.where(np.arange(Nkv)[None, :] <= pos, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)                    # pass 1
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)                    # pass 2
    p = e / l                                            # pass 3
    return np.einsum("bhij,bhjd->bhid", p, v), (m + np.log(l))[..., 0]


def merge_partials(o_part, lse_part):
    """Merge S block states over disjoint key ranges, taken in order s = 0, 1, ...
    with the block-wise update of page "tm_flash_attention_math" ("The
    block-wise update, and the full algorithm"): a block with log-sum-exp
    lse_s and normalised output o_s carries m_s = lse_s, l_s = 1, o~_s = o_s;
    m_new = max(m, m_s), alpha = exp(m - m_new), l = alpha l + exp(m_s - m_new),
    o~ = alpha o~ + exp(m_s - m_new) o_s; finally o = o~ / l, lse = m + ln l.
    A block with lse_s = -inf (no visible key) leaves the state unchanged.
    o_part [S, rows, d], lse_part [S, rows] -> o [rows, d], lse [rows]."""
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    S, rows, d = o_part.shape
    o = np.zeros((rows, d))
    lse = np.full(rows, -np.inf)
    for r in range(rows):
        m, l, ot = -np.inf, 0.0, np.zeros(d)
        for s_ in range(S):
            ms = lse_part[s_, r]
            if ms == -np.inf:
                continue
            m_new = max(m, ms)
            alpha = np.exp(m - m_new) if m != -np.inf else 0.0
            w = np.exp(ms - m_new)
            l = alpha * l + w
            ot = alpha * ot + w * o_part[s_, r]
            m = m_new
        if l > 0.0:
            o[r] = ot / l
            lse[r] = m + np.log(l)
    return o, lse


def softmax_rows(x):
    """y = softmax of each row of x [rows, cols] and lse = log sum exp per row, by
    the three passes of page "tm_flash_attention_math" ("Safe softmax"):
    m = max, l = sum exp(x - m), y = exp(x - m) / l.  A row of only -inf gives
    y = 0 and lse = -inf (nothing is visible)."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=1, keepdims=True)
    ok = np.isfinite(m[:, 0])
    e = np.exp(np.where(ok[:, None], x - np.where(ok[:, None], m, 0.0), -np.inf))
    l = e.sum(axis=1, keepdims=True)
    y = np.where(ok[:, None], e / np.where(l > 0, l, 1.0), 0.0)
    lse = np.where(ok, m[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return y, lse
