"""Exact scaled-dot-product attention in fp64 NumPy (TEST INFRASTRUCTURE ONLY).

The definition, from [QBank-36] part 2 and [FA-memory] part 1: for every batch
b and query head h, with key/value group g(h),

    S = scale * Q_{b,h} K_{b,g}^T            (N x N)
    P = softmax(S) row by row                (two passes: row max, then exp / sum)
    O = P V_{b,g}
    LSE_i = m_i + ln sum_j exp(S_ij - m_i)   (natural log, includes the scale)

Causal [Lecture, "GPU 显存和注意力瓶颈"]: query i sees key j iff j <= i.
Grouped-query attention [Lecture, "减少缓存表示并验证草稿"]: Hq query heads
share Hkv key/value heads; query head h reads kv head h // (Hq // Hkv), so
Hkv == Hq is ordinary multi-head attention and Hkv == 1 is multi-query
attention.

The backward pass is the plain calculus of the definition above (the pages
say only that it is recomputed from saved statistics, [Lecture] and [QBank-36]
part 7): with dO given,

    dV_g = sum_{h in g} P^T dO
    dP   = dO V_g^T
    dS   = P * (dP - rowsum(P * dP))
    dQ_h = scale * dS K_g
    dK_g = sum_{h in g} scale * dS^T Q_h

The implementation materialises full rows of S and P for a block of query
rows at a time.  Row blocking is an exact partition of independent rows, not
an online softmax, so every row is computed by the two-pass definition.
"""
from __future__ import annotations

import numpy as np

__all__ = ["attention_forward", "attention_backward", "kv_head_index",
           "visible_mask", "softmax_rows"]


def kv_head_index(h: int, Hq: int, Hkv: int) -> int:
    """Key/value head read by query head h: contiguous groups of Hq // Hkv heads."""
    return h // (Hq // Hkv)


def visible_mask(rows: np.ndarray, N: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), N]: True where query rows[r] may attend to key j."""
    cols = np.arange(N)
    if causal:
        return cols[None, :] <= rows[:, None]
    return np.ones((len(rows), N), dtype=bool)


def softmax_rows(s: np.ndarray):
    """Two-pass softmax of each row of s (masked entries are -inf).

    Returns (P, m, den) with m the row max and den = sum_j exp(s_ij - m_i).
    """
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    den = np.sum(e, axis=1, keepdims=True)
    return e / den, m[:, 0], den[:, 0]


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, Hq, N, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    Hkv = k.shape[1]
    if Hkv < 1 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, N, d


def _rows_of_p(q_blk, k_g, rows, N, causal, scale):
    s = scale * (q_blk @ k_g.T)
    s = np.where(visible_mask(rows, N, causal), s, -np.inf)
    return softmax_rows(s)


def _row_span(N, row_range):
    if row_range is None:
        return 0, N
    r0, r1 = row_range
    if not (0 <= r0 <= r1 <= N):
        raise ValueError("row_range outside [0, N]")
    return r0, r1


def attention_forward(q, k, v, causal: bool, scale: float, row_block: int = 512, row_range=None):
    """O [B,Hq,N,d] and LSE [B,Hq,N] of exact attention, in fp64.

    ``row_range=(r0, r1)`` computes only query rows r0..r1-1 (the other rows of
    the outputs are left as NaN); each row is still the full two-pass softmax
    over every key, so a row range is a bounded sample of the same work.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    lo, hi = _row_span(N, row_range)
    o = np.full((B, Hq, N, d), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_index(h, Hq, Hkv)
            for r0 in range(lo, hi, row_block):
                r1 = min(hi, r0 + row_block)
                rows = np.arange(r0, r1)
                p, m, den = _rows_of_p(q[b, h, r0:r1], k[b, g], rows, N, causal, scale)
                o[b, h, r0:r1] = p @ v[b, g]
                lse[b, h, r0:r1] = m + np.log(den)
    return o, lse


def attention_backward(q, k, v, do, causal: bool, scale: float, row_block: int = 512, row_range=None):
    """(dQ, dK, dV) of L = sum(dO * O) for exact attention, in fp64.

    ``row_range=(r0, r1)`` restricts the sum to query rows r0..r1-1: dQ rows
    outside it are zero and dK/dV hold only those rows' contributions.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Hq, Hkv, N, d = _check_shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("dO must match q")
    dq = np.zeros((B, Hq, N, d))
    dk = np.zeros((B, Hkv, N, d))
    dv = np.zeros((B, Hkv, N, d))
    lo, hi = _row_span(N, row_range)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_index(h, Hq, Hkv)
            for r0 in range(lo, hi, row_block):
                r1 = min(hi, r0 + row_block)
                rows = np.arange(r0, r1)
                q_blk = q[b, h, r0:r1]
                do_blk = do[b, h, r0:r1]
                p, _, _ = _rows_of_p(q_blk, k[b, g], rows, N, causal, scale)
                dv[b, g] += p.T @ do_blk
                dp = do_blk @ v[b, g].T
                ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
                dq[b, h, r0:r1] = scale * (ds @ k[b, g])
                dk[b, g] += scale * (ds.T @ q_blk)
    return dq, dk, dv
