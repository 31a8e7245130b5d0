"""Seeded synthetic inputs and the workload table.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can be fed
from it.  Every tensor is drawn in fp32 on the CPU from a ``torch.Generator``
seeded with the workload's seed, in the fixed order Q, K, V, dO, and then
rounded to bf16.  The oracle receives the same bf16 values upcast to fp64, so
input quantisation is never counted as kernel error.

Distributions follow the workloads: Q, K, V, dO ~ N(0, 1), except the
logit-stress workload, where Q ~ 4 N(0, 1) (scores with standard deviation 4,
so the running maximum keeps rising late in a row) and V ~ U(-1, 1).
"""
import math

import torch

# name -> shape, causal modes, passes, distribution knobs, seed.
# "slice" marks the reduced case on which the long-sequence backward is checked.
WORKLOADS = {
    "single_head_n256_d64": dict(B=1, H=1, N=256, d=64, causal=(False,), passes=("fwd",),
                                 q_std=1.0, v_dist="normal", seed=1235),
    "b4h16_n2048_d64": dict(B=4, H=16, N=2048, d=64, causal=(False, True), passes=("fwd", "bwd"),
                            q_std=1.0, v_dist="normal", seed=1236),
    "b1h32_n8192_d128_causal": dict(B=1, H=32, N=8192, d=128, causal=(True,), passes=("fwd", "bwd"),
                                    q_std=1.0, v_dist="normal", seed=1237),
    "logit_stress_b2h16_n4000_d128": dict(B=2, H=16, N=4000, d=128, causal=(False,), passes=("fwd",),
                                          q_std=4.0, v_dist="uniform", seed=1238),
    "long_b1h16_n32768_d128_causal": dict(B=1, H=16, N=32768, d=128, causal=(True,),
                                          passes=("fwd", "bwd"), q_std=1.0, v_dist="normal", seed=1239),
    "long_bwd_slice_b1h1_n4096_d128_causal": dict(B=1, H=1, N=4096, d=128, causal=(True,),
                                                  passes=("bwd",), q_std=1.0, v_dist="normal",
                                                  seed=1240),
}

HEADLINE = "b1h32_n8192_d128_causal"


def default_scale(d):
    """1/sqrt(d), the scale every workload uses."""
    return 1.0 / math.sqrt(d)


def make_inputs(B, H, N, d, seed, q_std=1.0, v_dist="normal", with_do=False):
    """Return bf16 CPU tensors (q, k, v[, do]) of shape [B, H, N, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32) * float(q_std)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    if v_dist == "normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif v_dist == "uniform":
        v = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(v_dist)
    out = [q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)]
    if with_do:
        out.append(torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16))
    return tuple(out)


def workload_inputs(name, with_do=False, **override):
    """Inputs for a named workload; ``override`` may replace B, H, N, d or seed."""
    w = dict(WORKLOADS[name])
    w.update(override)
    return make_inputs(w["B"], w["H"], w["N"], w["d"], w["seed"], w["q_std"], w["v_dist"], with_do)


def sample_rows(N, count, seed, always=(0, 127, 128)):
    """Seeded query-row sample of min(count, N) distinct rows: the listed rows,
    N-1, then uniform draws (repeated draws are drawn again)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    rows = set(r for r in always if r < N) | {N - 1}
    count = min(count, N)
    while len(rows) < count:
        rows.update(torch.randint(0, N, (count - len(rows),), generator=g).tolist())
    return sorted(rows)[:count] if len(rows) > count else sorted(rows)


def make_varlen_inputs(lengths, H, d, seed, with_do=False):
    """Packed variable-length batch: bf16 CPU tensors (q, k, v[, do]) of shape
    [H, T, d] (sequence b at rows [cu[b], cu[b+1]) of every head, T = sum of
    lengths) and the int32 offsets cu [B + 1].  Values ~ N(0, 1), drawn in fp32
    in the order Q, K, V, dO."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    T = int(sum(lengths))
    shape = (H, T, d)
    out = [torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
           for _ in range(4 if with_do else 3)]
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return tuple(out) + (cu,)


def varlen_lengths(B, lo, hi, seed):
    """B sequence lengths drawn uniformly from [lo, hi] (a seeded length mix)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


# Packed variable-length workloads (profiling; not one of the fixed-shape
# workloads above): B sequences with lengths drawn uniformly from [lo, hi].
VARLEN_WORKLOADS = {
    "varlen_b16h16_len512to8192_d128_causal": dict(B=16, H=16, d=128, lo=512, hi=8192,
                                                   seed=1241, causal=True),
}


# Decoding workloads (profiling): Nq queries at the end of Nkv keys, Q, K, V ~ N(0, 1).
DECODE_WORKLOADS = {
    "decode_b4h32_nq1_nkv32768_d128": dict(B=4, H=32, Nq=1, Nkv=32768, d=128, seed=1242,
                                           causal=True),
}


# Row-softmax workloads (profiling): fp32 rows ~ 30 N(0, 1).
SOFTMAX_WORKLOADS = {
    "softmax_rows4096_cols32768_f32": dict(rows=4096, cols=32768, seed=1243),
}


def make_softmax_input(rows, cols, seed, scale=30.0):
    """fp32 CPU tensor [rows, cols] ~ scale * N(0, 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn((rows, cols), generator=g, dtype=torch.float32) * float(scale)


# Host-CPU workloads (the flash-style forward on the host cores): fp32 inputs
# drawn like make_inputs (N(0, 1), order Q, K, V, rounded to bf16 and widened
# back, so the values are the same kind the GPU path sees).  The shape is a
# small-model attention layer at a long context: 16 heads of d = 64, 4096 tokens.
HOST_WORKLOADS = {
    "host_b1h16_n4096_d64_causal": dict(B=1, H=16, N=4096, d=64, seed=1244, causal=True),
}


def make_host_inputs(B, H, N, d, seed, q_std=1.0, v_dist="normal"):
    """fp32 numpy arrays (q, k, v) of shape [B, H, N, d] (bf16-representable values)."""
    return tuple(t.float().numpy() for t in make_inputs(B, H, N, d, seed, q_std, v_dist))
