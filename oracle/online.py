"""The pages' streaming softmax-weighted sum (TEST INFRASTRUCTURE ONLY).

[Lecture, "推导 FlashAttention 的在线 softmax"] writes one query's attention
output as a numerator (sum of exp(score) * value) over a denominator (sum of
exp(score)), accumulated as (score, value) pairs arrive.  To stay stable, both
sums are kept relative to the largest score seen so far: the first element's
reference is its own score, and whenever a later score raises the running
maximum, the accumulated numerator and denominator are multiplied by
exp(old_max - new_max) before the new terms are added.  Multiplying both by
the same factor leaves their ratio unchanged, so the result is the exact
softmax-weighted sum.  [QBank-36] part 3 does the same per tile of keys.

This is the algorithm in the order the pages give it, kept separate from the
two-pass definition in ``oracle.ref`` so that each pins the other.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence


def stream(scores: Sequence[float], values: Sequence, block: int = 1, trace=None):
    """Stream (score, value) pairs in blocks of ``block``.

    ``values`` holds scalars or equal-length sequences.  Returns
    (numerator, denominator, running_max).  If ``trace`` is a list, the state
    (m, numerator, denominator) after every block is appended to it.
    """
    n = len(scores)
    if n == 0:
        raise ValueError("empty row")
    vec = not isinstance(values[0], (int, float))
    width = len(values[0]) if vec else 1
    m = -math.inf
    num = [0.0] * width
    den = 0.0
    for start in range(0, n, block):
        blk_s = scores[start:start + block]
        blk_v = values[start:start + block]
        m_new = max(m, max(blk_s))
        factor = math.exp(m - m_new) if m != -math.inf else 0.0
        num = [x * factor for x in num]
        den = den * factor
        for s, v in zip(blk_s, blk_v):
            w = math.exp(s - m_new)
            den += w
            if vec:
                num = [x + w * vc for x, vc in zip(num, v)]
            else:
                num[0] += w * v
        m = m_new
        if trace is not None:
            trace.append((m, num[0] if not vec else list(num), den))
    return (num if vec else num[0]), den, m


def softmax_weighted_sum(scores: Sequence[float], values: Sequence, block: int = 1):
    """Numerator / denominator of ``stream``: the softmax-weighted sum of values."""
    num, den, m = stream(scores, values, block)
    if isinstance(num, list):
        return [x / den for x in num]
    return num / den


def log_sum_exp(scores: Iterable[float], block: int = 1) -> float:
    """ln sum exp(scores), from the streamed running max and denominator."""
    s = list(scores)
    _, den, m = stream(s, [0.0] * len(s), block)
    return m + math.log(den)
