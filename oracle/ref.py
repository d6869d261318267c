"""Exact scaled-dot-product attention in fp64 NumPy (TEST INFRASTRUCTURE ONLY).

The definition, from [QBank-36] part 2 and [FA-memory] part 1: for every batch
b and query head h, with key/value group g(h),

    S = scale * Q_{b,h} K_{b,g}^T            (N x N)
    P = softmax(S) row by row                (two passes: row max, then exp / sum)
    O = P V_{b,g}
    LSE_i = m_i + ln sum_j exp(S_ij - m_i)   (natural log, includes the scale)

Causal [Lecture, "GPU 显存和注意力瓶颈"]: query i sees key j iff j <= i.
With fewer query rows than keys (Nq < Nk, the decode shape: a few new
queries against a long key/value history) query row i stands at position
i + (Nk - Nq), the last Nq positions, and causal visibility compares key
positions with that.  Sliding window ([ZeRO-vs-FA] "注意力瓶颈与优化路线" and
[FA-memory] part 2 name local windows as a different visibility pattern):
with window w >= 1 query position p sees key j iff p - w < j <= p; the window
is only defined together with causal visibility.
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
           "visible_mask", "softmax_rows", "query_positions", "merge_partials"]


def kv_head_index(h: int, Hq: int, Hkv: int) -> int:
    """Key/value head read by query head h: contiguous groups of Hq // Hkv heads."""
    return h // (Hq // Hkv)


def query_positions(rows: np.ndarray, Nq: int, Nk: int) -> np.ndarray:
    """Positions of query rows among the keys: the Nq queries are the last Nq
    positions (row i stands at i + Nk - Nq; i itself when Nq == Nk)."""
    return np.asarray(rows) + (Nk - Nq)


def visible_mask(pos: np.ndarray, N: int, causal: bool, window: int = 0) -> np.ndarray:
    """Boolean [len(pos), N]: True where the query at position pos[r] may attend
    to key j (j <= pos when causal; also j > pos - window when window > 0)."""
    cols = np.arange(N)
    if window and not causal:
        raise ValueError("a sliding window needs causal visibility")
    if causal:
        m = cols[None, :] <= pos[:, None]
        if window:
            m &= cols[None, :] > pos[:, None] - window
        return m
    return np.ones((len(pos), N), dtype=bool)


def softmax_rows(s: np.ndarray):
    """Two-pass softmax of each row of s (masked entries are -inf).

    Returns (P, m, den) with m the row max and den = sum_j exp(s_ij - m_i).
    """
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    den = np.sum(e, axis=1, keepdims=True)
    return e / den, m[:, 0], den[:, 0]


def _check_shapes(q, k, v, causal=False):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Nk, d] matching q")
    Hkv, Nk = k.shape[1], k.shape[2]
    if Hkv < 1 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if causal and Nq > Nk:
        raise ValueError("causal visibility needs Nq <= Nk")
    return B, Hq, Hkv, Nq, Nk, d


def _rows_of_p(q_blk, k_g, rows, Nq, causal, scale, window):
    Nk = k_g.shape[0]
    s = scale * (q_blk @ k_g.T)
    s = np.where(visible_mask(query_positions(rows, Nq, Nk), Nk, causal, window), s, -np.inf)
    return softmax_rows(s)


def _row_span(N, row_range):
    if row_range is None:
        return 0, N
    r0, r1 = row_range
    if not (0 <= r0 <= r1 <= N):
        raise ValueError("row_range outside [0, N]")
    return r0, r1


def attention_forward(q, k, v, causal: bool, scale: float, row_block: int = 512, row_range=None, window: int = 0):
    """O [B,Hq,Nq,d] and LSE [B,Hq,Nq] of exact attention, in fp64.

    ``row_range=(r0, r1)`` computes only query rows r0..r1-1 (the other rows of
    the outputs are left as NaN); each row is still the full two-pass softmax
    over every key, so a row range is a bounded sample of the same work.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Hkv, N, Nk, d = _check_shapes(q, k, v, causal)
    lo, hi = _row_span(N, row_range)
    o = np.full((B, Hq, N, d), np.nan)
    lse = np.full((B, Hq, N), np.nan)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_index(h, Hq, Hkv)
            for r0 in range(lo, hi, row_block):
                r1 = min(hi, r0 + row_block)
                rows = np.arange(r0, r1)
                p, m, den = _rows_of_p(q[b, h, r0:r1], k[b, g], rows, N, causal, scale, window)
                o[b, h, r0:r1] = p @ v[b, g]
                lse[b, h, r0:r1] = m + np.log(den)
    return o, lse


def attention_backward(q, k, v, do, causal: bool, scale: float, row_block: int = 512, row_range=None,
                       window: int = 0, o_for_d=None):
    """(dQ, dK, dV) of L = sum(dO * O) for exact attention, in fp64.

    ``row_range=(r0, r1)`` restricts the sum to query rows r0..r1-1: dQ rows
    outside it are zero and dK/dV hold only those rows' contributions.

    ``o_for_d``: the backward recomputes from what the forward saved (the
    output O and the log-sum-exp), so D_i = rowsum(P * dP) can be formed as
    rowsum(dO * O), the same number in exact arithmetic (O = P V, so
    dO_i . O_i = sum_j P_ij dO_i . v_j = sum_j P_ij dP_ij).  Given an O
    [B, Hq, N, d] here (e.g. the forward's output rounded to bf16), D is
    formed from it; by default D = rowsum(P * dP) from the exact P.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Hq, Hkv, N, Nk, d = _check_shapes(q, k, v, causal)
    if do.shape != q.shape:
        raise ValueError("dO must match q")
    dq = np.zeros((B, Hq, N, d))
    dk = np.zeros((B, Hkv, Nk, d))
    dv = np.zeros((B, Hkv, Nk, d))
    lo, hi = _row_span(N, row_range)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_index(h, Hq, Hkv)
            for r0 in range(lo, hi, row_block):
                r1 = min(hi, r0 + row_block)
                rows = np.arange(r0, r1)
                q_blk = q[b, h, r0:r1]
                do_blk = do[b, h, r0:r1]
                p, _, _ = _rows_of_p(q_blk, k[b, g], rows, N, causal, scale, window)
                dv[b, g] += p.T @ do_blk
                dp = do_blk @ v[b, g].T
                if o_for_d is None:
                    drow = np.sum(p * dp, axis=1, keepdims=True)
                else:
                    drow = np.sum(do_blk * np.asarray(o_for_d[b, h, r0:r1], dtype=np.float64), axis=1, keepdims=True)
                ds = p * (dp - drow)
                dq[b, h, r0:r1] = scale * (ds @ k[b, g])
                dk[b, g] += scale * (ds.T @ q_blk)
    return dq, dk, dv


def merge_partials(o_parts, lse_parts):
    """Combine attention over disjoint key subsets into attention over their union.

    Part s holds O_s (normalised within its keys) and LSE_s = ln sum_{j in s}
    exp(S_ij); a part with no visible key has LSE_s = -inf and is ignored.
    Following [Lecture] "推导 FlashAttention 的在线 softmax" -- numerator and
    denominator carried relative to a reference maximum and rescaled by
    exp(old - new) when that reference changes -- each part's numerator is
    exp(LSE_s) O_s and its denominator exp(LSE_s); both are taken relative to
    m = max_s LSE_s, summed, and divided:

        O = sum_s exp(LSE_s - m) O_s / sum_s exp(LSE_s - m),
        LSE = m + ln sum_s exp(LSE_s - m).

    o_parts: [S, ..., d]; lse_parts: [S, ...].
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    w = np.exp(lse_parts - m[None])
    den = np.sum(w, axis=0)
    num = np.sum(np.where(w[..., None] > 0, w[..., None] * o_parts, 0.0), axis=0)
    return num / den[..., None], m + np.log(den)
