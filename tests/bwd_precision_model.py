"""A CPU model of the backward kernel's number formats, used only to DERIVE
tolerances for the parity tests.  It is not an oracle: the oracle
(``oracle.attention_bwd``) is the fp64 reference every result is compared
with, and this model shares no code with it or with the CUDA path.

The pages fix no precisions for the backward pass ("FlashAttention tiles
exact softmax without materializing the score matrix", "Backward computation
can trade recomputation for stored intermediates").  The library's kernels
round at these points, and the model rounds at the same ones:

  forward   O rounded to bf16; LSE kept in fp32 (natural log)
  D_i       sum_c dO_ic O_ic in fp32, from the bf16 O
  P         exp2(S scale log2e - LSE log2e) in fp32, rounded to bf16 once;
            the same bf16 P feeds dV and dS
  dP        dO V^T accumulated in fp32
  dS        P (dP - D) formed in fp32 from the bf16 P, rounded to bf16
  dV, dK, dQ  P^T dO, scale dS^T Q, scale dS K accumulated in fp32, rounded
            to bf16 at the output

Every matmul has exact products of bf16 inputs and fp32 sums.  With
``exact=True`` nothing is rounded and everything is fp64: the model then
computes the oracle's gradients, which a CPU test checks.

Two fp32 evaluations that are both faithful to these formats (another
summation order, ex2.approx instead of exp2, the forward's own LSE) differ by
a few units in the last place of fp32, and that is enough to flip individual
bf16 roundings of P and dS.  ``derived_bars`` measures that spread by
re-running the model with its fp32 intermediates scaled by (1 + u 2^-20),
u uniform in [-1, 1] (about eight fp32 ulps).  With x_r the fp32 output of
run r BEFORE its final bf16 rounding (x_0 unperturbed) and ref the fp64
oracle, a kernel output g = bf16(x_k) satisfies

    |g - ref| <= |x_0 - ref| + |x_k - x_0| + half_ulp_bf16(|x_k|)

so the bar of each tensor is, over its elements e,

    G   = 1.25 max_r max_e |x_r - x_0|          (spread of valid evaluations,
                                                 a quarter added because the
                                                 kernel is one more sample)
    bar = max_e ( |x_0 - ref| + half_ulp_bf16(|ref| + |x_0 - ref| + G) ) + G
"""
import numpy as np

L2E = 1.4426950408889634


def bf16_round(x):
    """Round float32 values to bfloat16 (to nearest, ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _jitter(x, rng, rel):
    if rng is None:
        return x
    return (x * (1.0 + rel * rng.uniform(-1.0, 1.0, x.shape))).astype(x.dtype)


def half_ulp_bf16(a):
    """Half a bfloat16 unit in the last place at magnitude a (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(a, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8.0)


def backward(q, k, v, do, scale, causal, exact=False, rng=None, rel=2.0 ** -20, raw=False):
    """dQ, dK, dV [B,H,N,d] (float64 arrays) of softmax(scale Q K^T) V for
    dL/dO = do, evaluated in the kernel's number formats (or exactly).  With
    ``raw`` the outputs are returned before their final bf16 rounding."""
    B, H, N, d = q.shape
    ft = np.float64 if exact else np.float32
    rnd = (lambda x: x) if exact else bf16_round
    jit = (lambda x: x) if exact else (lambda x: _jitter(x, rng, rel))
    outs = [np.empty((B * H, N, d)) for _ in range(3)]
    mask = np.triu(np.ones((N, N), dtype=bool), 1) if causal else np.zeros((N, N), dtype=bool)
    sl2 = ft(scale) * ft(L2E)
    for bh in range(B * H):
        Q, K, V, dO = (np.asarray(x, dtype=np.float64).reshape(B * H, N, d)[bh].astype(ft)
                       for x in (q, k, v, do))
        S = jit(Q @ K.T)
        # forward: O and LSE as the forward kernel leaves them
        z = np.where(mask, -np.inf, S * sl2).astype(ft)
        m = z.max(axis=1, keepdims=True)
        e = np.exp2(z - m).astype(ft)
        l = e.sum(axis=1, keepdims=True, dtype=ft)
        O = rnd(jit((e @ V) / l))
        lse = ((m[:, 0] + np.log2(l[:, 0])) / ft(L2E)).astype(ft)
        # backward
        Dl = jit((dO * O).sum(axis=1, dtype=ft))
        P = rnd(jit(np.exp2(np.where(mask, -np.inf, S * sl2 - lse[:, None] * ft(L2E))).astype(ft)))
        dP = jit(dO @ V.T)
        dS = rnd(jit((P * (dP - Dl[:, None])).astype(ft)))
        out_rnd = (lambda x: x) if raw else rnd
        outs[2][bh] = out_rnd(jit(P.T @ dO))
        outs[1][bh] = out_rnd(jit(ft(scale) * (dS.T @ Q)))
        outs[0][bh] = out_rnd(jit(ft(scale) * (dS @ K)))
    return tuple(o.reshape(B, H, N, d) for o in outs)


def derived_bars(q, k, v, do, scale, causal, ref, runs=8, seed=0):
    """Per-tensor max-abs bars (dQ, dK, dV) for a kernel result against the
    fp64 reference ``ref`` (the rule in the module docstring), and the mean-abs
    errors of the model's rounded outputs."""
    rng = np.random.default_rng(seed)
    base = backward(q, k, v, do, scale, causal, raw=True)
    sims = [backward(q, k, v, do, scale, causal, rng=rng, raw=True) for _ in range(runs - 1)]
    rounded = backward(q, k, v, do, scale, causal)
    bars, means = [], []
    for t in range(3):
        G = 1.25 * max(float(np.abs(s[t] - base[t]).max()) for s in sims)
        err0 = np.abs(base[t] - ref[t])
        bars.append(float((err0 + half_ulp_bf16(np.abs(ref[t]) + err0 + G)).max()) + G)
        means.append(float(np.abs(rounded[t] - ref[t]).mean()))
    return bars, means
