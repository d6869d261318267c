"""Exact attention in pure-Python loops, for tiny shapes (TEST INFRASTRUCTURE ONLY).

The same definition as ``oracle.ref`` (see there for the page citations),
written element by element with ``math.exp`` and no array library, so that
the vectorised oracle can be checked against an independent transcription.
Inputs are nested lists (or anything indexable) [B][H][N][d].
"""
from __future__ import annotations

import math


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def _keys(i, N, Nk, causal, window):
    # Query row i stands at position i + Nk - N (the last N of Nk positions).
    p = i + Nk - N
    return [j for j in range(Nk) if (not causal or (j <= p and (window == 0 or j > p - window)))]


def forward(q, k, v, causal: bool, scale: float, window: int = 0):
    """Return (o, lse) as nested lists."""
    B, Hq, N, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Nk = len(k[0]), len(k[0][0])
    group = Hq // Hkv
    o = [[[[0.0] * d for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * N for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(N):
                keys = _keys(i, N, Nk, causal, window)
                s = [scale * _dot(q[b][h][i], k[b][g][j]) for j in keys]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                den = sum(w)
                for c in range(d):
                    o[b][h][i][c] = sum(w[t] * v[b][g][j][c] for t, j in enumerate(keys)) / den
                lse[b][h][i] = m + math.log(den)
    return o, lse


def backward(q, k, v, do, causal: bool, scale: float, window: int = 0):
    """Return (dq, dk, dv) as nested lists, element by element."""
    B, Hq, N, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv, Nk = len(k[0]), len(k[0][0])
    group = Hq // Hkv
    dq = [[[[0.0] * d for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    dk = [[[[0.0] * d for _ in range(Nk)] for _ in range(Hkv)] for _ in range(B)]
    dv = [[[[0.0] * d for _ in range(Nk)] for _ in range(Hkv)] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(N):
                keys = _keys(i, N, Nk, causal, window)
                s = [scale * _dot(q[b][h][i], k[b][g][j]) for j in keys]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                den = sum(w)
                p = [x / den for x in w]
                dp = [_dot(do[b][h][i], v[b][g][j]) for j in keys]
                pdp = sum(pi * dpi for pi, dpi in zip(p, dp))
                for t, j in enumerate(keys):
                    ds = p[t] * (dp[t] - pdp)
                    for c in range(d):
                        dv[b][g][j][c] += p[t] * do[b][h][i][c]
                        dq[b][h][i][c] += scale * ds * k[b][g][j][c]
                        dk[b][g][j][c] += scale * ds * q[b][h][i][c]
    return dq, dk, dv
