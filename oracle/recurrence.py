"""Scalar model of the online-softmax recurrence, in fp64.  TEST INFRASTRUCTURE ONLY.

Only tests/ may import this module.  It restates, for a single query, the
block-wise algorithm of "tm_flash_attention_math" (page 3, "The block-wise
update, and the full algorithm"): carry a running maximum m, a running
denominator l and an unnormalised output o~; for each block of keys take the
block maximum, rescale the old state by alpha = exp(m_old - m_new) and add the
block's terms measured against m_new; divide by l once at the end.  The same
recurrence, for l alone, is page 1's "Online softmax carries a maximum and a
normalizer" and the eight-score table of "Decoding flash attention".

The model exists to pin the pages' worked examples and invariants (stability:
every exp argument <= 0; exactness: block size and order do not change the
result).  ``slack`` > 0 keeps the old reference m unless a block raises the
maximum by more than ``slack``: the page's shift invariance ("for ANY constant
m", section "Safe softmax: the max-subtraction we cannot give up") says the
result is unchanged, and every exp argument stays <= slack instead of <= 0.  The ``pitfall`` switch plants, on purpose, each of the four mistakes
listed under page 3's "Pitfalls in implementing the recurrence", so that tests
can show the checks catch them:

  "rescale_l_only"      o~ is not multiplied by alpha
  "finite_m_init"       m starts at 0.0 instead of -inf
  "mask_after_max"      the block maximum is taken before masked scores are
                        set to -inf
  "normalize_per_block" o~ is divided by l after every block
"""
import math

PITFALLS = ("rescale_l_only", "finite_m_init", "mask_after_max", "normalize_per_block")


def _axpy(alpha, x, y):
    return [alpha * a + b for a, b in zip(x, y)]


def online_softmax_attention(scores, values, blocks, visible=None, pitfall=None, slack=0.0):
    """Run the block-wise recurrence for one query.

    scores  -- list of raw scaled scores s_j (floats)
    values  -- list of value vectors v_j (each a list of floats)
    blocks  -- list of lists of key indices, visited in the given order
    visible -- optional list of bools; False marks a masked key (causal or padding)
    pitfall -- None or one of PITFALLS
    slack   -- 0 for the page's algorithm (m is the running max); > 0 moves m
               only when the block maximum exceeds it by more than ``slack``

    Returns (o, m, l, trace).  trace is one dict per block with the block
    maximum, m_new, alpha, the p_j, l, o~ and every exp argument used.
    """
    if pitfall is not None and pitfall not in PITFALLS:
        raise ValueError(pitfall)
    dv = len(values[0])
    m = 0.0 if pitfall == "finite_m_init" else -math.inf
    l = 0.0
    o_t = [0.0] * dv
    trace = []
    for block in blocks:
        vis = [True if visible is None else bool(visible[j]) for j in block]
        raw = [float(scores[j]) for j in block]
        masked = [s if ok else -math.inf for s, ok in zip(raw, vis)]
        m_blk = max(raw) if pitfall == "mask_after_max" else max(masked)
        m_new = max(m, m_blk)
        if slack > 0 and m != -math.inf and m_new - m <= slack:
            m_new = m  # keep the old reference
        args = []
        if m_new == -math.inf:
            # nothing visible yet: exp(-inf - (-inf)) is undefined; the state stays empty
            alpha, p = 1.0, [0.0] * len(block)
        else:
            args.append(m - m_new)
            alpha = math.exp(m - m_new)
            p = []
            for s in masked:
                args.append(s - m_new)
                p.append(math.exp(s - m_new))
        l_old = l
        l = alpha * l + sum(p)
        contrib = [0.0] * dv
        for pj, j in zip(p, block):
            contrib = _axpy(pj, values[j], contrib)
        if pitfall == "rescale_l_only":
            o_t = [a + b for a, b in zip(o_t, contrib)]
        else:
            o_t = _axpy(alpha, o_t, contrib)
        if pitfall == "normalize_per_block" and l > 0:
            o_t = [x / l for x in o_t]
        m = m_new
        trace.append(dict(m_blk=m_blk, m_new=m_new, alpha=alpha, p=p, l_old=l_old, l=l,
                          o_tilde=list(o_t), exp_args=args))
    o = [x / l for x in o_t] if l > 0 else [math.nan] * dv
    return o, m, l, trace


def blocks_of(n, size, order=None):
    """Split key indices 0..n-1 into consecutive blocks of ``size``; optionally
    visit the blocks in the permuted ``order``."""
    blocks = [list(range(s, min(s + size, n))) for s in range(0, n, size)]
    if order is not None:
        blocks = [blocks[i] for i in order]
    return blocks
