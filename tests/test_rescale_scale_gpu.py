"""GPU parity (through the C ABI, against the fp64 oracle) on inputs that make
the online softmax rescale for real, and with softmax scales away from 1/sqrt(d).

The running-max rescale ([Lecture] "推导 FlashAttention 的在线 softmax": when a
row's maximum grows, the running numerator and denominator are multiplied by
exp(old max - new max)) only changes the kernel's state when a row's maximum
climbs by more than the forward kernel's lazy threshold of 24 log2 units after
the first key tile of a work item.  N(0, 1) scores never do that, so here the
scores are given planted steps: query column 0 is set to a constant A and key
column 0 of key tile T to beta_T, which adds scale * A * beta_T to every score
against that tile.  The steps are chosen from the other columns' score spread
so that every row's maximum jumps by more than the threshold, and
``rescale_events`` checks that claim on the CPU from the bf16 inputs before
the GPU result is compared.

A is large (128) so that beta stays small: column 0 of dQ = scale * dS K is
scale * sum_j dS_ij beta(j), and since every row of dS sums to zero it is a
near-total cancellation whose exact value is tiny, while the bf16 rounding of
the dS operand (which the tolerances allow) contributes about beta * 2^-9 of
|dS| to it.  With A = 4 (beta up to ~500) that alone puts dQ's relative L2
error near 0.07 for any bf16-operand kernel (a CPU emulation of the
operand roundings gives the same); with A = 128 it is ~0.003.  Patterns:

  every  -- each key tile one step above the last, so every later tile of an
            item rescales: two consecutive tiles (both softmax groups), the
            item's last tile (the cross-group row-sum combine) and, under causal
            masking, the diagonal tile;
  mixed  -- full steps at tiles 1, 2, 5 and the last tile, half a step (below
            the threshold: the reference max lags and the probabilities exceed
            1) at tile 3.

The scale cases run plain, deterministic-backward and key-split paths with
scale in {0.05, 0.3, 1.0}, so a kernel that assumed 1/sqrt(d) anywhere (the
dK write-out, the dQ conversion, the deterministic dQ kernel, the split merge)
would fail.  At these scales many rows are dominated by one key, so O is
close to one V row (|O| up to ~4.5), and the bf16 rounding of the output alone
is up to half an ulp, 0.0156 for values in [4, 8): these are the cases where
the forward's correction for the rounding of each tile's largest weight
matters (without it a CPU emulation of the kernel's arithmetic gives max-abs
0.0275 at scale 0.3, with it 0.0095).  Outputs are written into buffers with guard bytes on both sides,
checked to be intact afterwards.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300.inputs import make_qkvdo
from oracle import ref
from tests.parity import GuardedBuffers, assert_bwd, assert_fwd

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
THRESHOLD_LOG2 = 24.0     # the forward kernel's lazy-rescale threshold (log2 units)
LOG2E = 1.0 / math.log(2.0)
A_COL0 = 128.0            # query column 0 (see the module docstring)


def f64(t):
    return t.double().numpy()


def gen(B, Hq, Hkv, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Nq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Nk, d), generator=g).to(torch.bfloat16)
    do = torch.randn((B, Hq, Nq, d), generator=g).to(torch.bfloat16)
    return q, k, v, do


def plant_steps(q, k, scale, pattern):
    """Set q[..., 0] = A and k[..., tile T rows, 0] = beta_T (in place) so that
    scores against tile T rise by about offset_T nats over tile 0."""
    d = q.shape[-1]
    Nk = k.shape[2]
    ntk = (Nk + 127) // 128
    spread = 7.0 * scale * math.sqrt(d - 1)             # about +-3.5 sigma of the other columns
    step = THRESHOLD_LOG2 / LOG2E + spread + 3.0          # nats
    if pattern == "every":
        inc = [0.0] + [1.0] * (ntk - 1)
    elif pattern == "mixed":
        inc = [0.0] * ntk
        for t, a in ((1, 1.0), (2, 1.0), (3, 0.5), (5, 1.0), (ntk - 1, 1.0)):
            if 0 < t < ntk:
                inc[t] = a
    else:
        raise ValueError(pattern)
    off = np.cumsum(inc) * step
    q[..., 0] = A_COL0
    for t in range(ntk):
        k[:, :, t * 128:(t + 1) * 128, 0] = off[t] / (scale * A_COL0)
    return q, k


def item_ranges(Nq, Nk, causal, window, splits, qpos_lo, qpos_hi):
    """Key-tile ranges [lo, hi) of the forward's work items for a query tile
    whose rows stand at positions qpos_lo..qpos_hi (each split is an item)."""
    ntk = (Nk + 127) // 128
    hi = min(ntk, qpos_hi // 128 + 1) if causal else ntk
    lo = max(0, qpos_lo - window + 1) // 128 if window > 0 else 0
    if splits <= 1:
        return [(lo, hi)] if hi > lo else []
    st = -(-ntk // splits)
    out = []
    for s in range(-(-ntk // st)):
        a, b = max(lo, s * st), min(hi, (s + 1) * st)
        if b > a:
            out.append((a, b))
    return out


def rescale_events(q, k, scale, causal, window=0, splits=1, packed_rows=None):
    """Count, on the CPU in fp64 from the bf16 inputs, the (row, item, tile)
    places where a row's tile maximum exceeds the maximum of every earlier
    tile of its item by more than the threshold + 1 log2 unit, so the kernel
    must rescale there with 0 < alpha < 1.  Returns (events, rows, rows with an
    event at an item's last tile, rows with events at two consecutive tiles)."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    qq, kk = f64(q), f64(k)
    ev = rows_ev = last_ev = consec_ev = 0
    tile_rows = packed_rows or 128
    for b in range(B):
        for h in range(Hq):
            s = scale * (qq[b, h] @ kk[b, h // G].T) * LOG2E       # [Nq, Nk] log2 units
            pos = np.arange(Nq) + (Nk - Nq)
            vis = ref.visible_mask(pos, Nk, causal, window)
            s = np.where(vis, s, -np.inf)
            for t0 in range(0, Nq, tile_rows):
                rr = np.arange(t0, min(Nq, t0 + tile_rows))
                if packed_rows:
                    lo_p, hi_p = Nk - Nq, Nk - 1
                else:
                    lo_p, hi_p = pos[rr[0]], pos[rr[-1]]
                for lo, hi in item_ranges(Nq, Nk, causal, window, splits, lo_p, hi_p):
                    tm = np.stack([s[rr, j * 128:(j + 1) * 128].max(axis=1) for j in range(lo, hi)], 1)
                    run = np.maximum.accumulate(tm, axis=1)
                    prev = run[:, :-1]
                    hit = np.isfinite(prev) & (tm[:, 1:] > prev + THRESHOLD_LOG2 + 1.0)
                    ev += int(hit.sum())
                    rows_ev += int(hit.any(axis=1).sum())
                    if hit.shape[1]:
                        last_ev += int(hit[:, -1].sum())
                        consec_ev += int((hit[:, 1:] & hit[:, :-1]).any(axis=1).sum())
    return ev, rows_ev, last_ev, consec_ev


def fwd_bwd(q, k, v, do, causal, scale, window=0, deterministic=False, guards=None):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    B, Hq, N, d = q.shape
    g = guards or GuardedBuffers(DEV)
    o = g.empty(q.shape, torch.bfloat16)
    lse = g.empty((B, Hq, N), torch.float32)
    if window:
        fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, window=window, out=o, lse=lse)
    else:
        fa.forward(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse)
    dq, dk, dv = g.empty(q.shape, torch.bfloat16), g.empty(k.shape, torch.bfloat16), g.empty(k.shape, torch.bfloat16)
    fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, window=window, deterministic=deterministic,
                dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    fa.check_device_status()
    g.check()
    return o, lse, dq, dk, dv


PLANTED = [
    # B, Hq, Hkv, N, d, causal, scale, pattern, window, deterministic
    (1, 2, 1, 1000, 128, True, 128 ** -0.5, "every", 0, False),
    (1, 2, 2, 900, 64, False, 64 ** -0.5, "mixed", 0, False),
    (2, 2, 1, 777, 64, True, 0.3, "every", 0, True),
    (1, 2, 1, 640, 128, False, 0.05, "mixed", 0, False),
    (1, 2, 2, 1000, 128, True, 128 ** -0.5, "every", 300, False),
    (1, 4, 2, 1100, 64, True, 64 ** -0.5, "mixed", 400, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,scale,pattern,window,det", PLANTED)
def test_running_max_rescale_forward_backward(cuda_lib, B, Hq, Hkv, N, d, causal, scale, pattern, window, det):
    q, k, v, do = gen(B, Hq, Hkv, N, N, d, seed=N + d + window)
    q, k = plant_steps(q, k, scale, pattern)
    ev, rows, last, consec = rescale_events(q, k, scale, causal, window)
    # Every query tile past the first (causal) or every tile (otherwise) holds
    # rows that must rescale; "every" also rescales at consecutive tiles and
    # at each item's last tile.
    assert rows >= B * Hq * (N - 128) * 0.9, (ev, rows)
    if pattern == "every":
        assert last > 0 and consec > 0, (ev, rows, last, consec)
    o, lse, dq, dk, dv = fwd_bwd(q, k, v, do, causal, scale, window, det)
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale, window=window)
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, scale, window=window)
    what = f"planted {pattern} N={N} d={d} causal={causal} scale={scale:.3g} window={window}"
    e = assert_fwd(o, lse, ro, rl, what)
    gr = assert_bwd(dq, dk, dv, rdq, rdk, rdv, what)
    print(what, "events", ev, e, gr)


@pytest.mark.parametrize("causal,splits,d,pattern", [(False, 3, 64, "every"), (True, 2, 128, "mixed"),
                                                     (False, 5, 128, "every")])
def test_running_max_rescale_key_splits(cuda_lib, causal, splits, d, pattern):
    B, Hq, Hkv, N = 2, 2, 1, 1100
    scale = d ** -0.5
    q, k, v, _ = gen(B, Hq, Hkv, N, N, d, seed=300 + splits)
    q, k = plant_steps(q, k, scale, pattern)
    ev, rows, _, _ = rescale_events(q, k, scale, causal, 0, splits)
    assert ev > 0 and rows > B * Hq * N * 0.5, (ev, rows)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale)
    assert_fwd(o, lse, ro, rl, f"planted {pattern}, {splits} splits")


@pytest.mark.parametrize("splits", [1, 3])
def test_running_max_rescale_packed_decode(cuda_lib, splits):
    # Grouped heads packed into one tile (4 heads x 3 rows), few queries
    # against 1000 keys: one item per (batch, kv head) and split.
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 3, 1000, 128
    scale = d ** -0.5
    q, k, v, _ = gen(B, Hq, Hkv, Nq, Nk, d, seed=500 + splits)
    q, k = plant_steps(q, k, scale, "every")
    ev, rows, last, consec = rescale_events(q, k, scale, True, 0, splits, packed_rows=Nq)
    assert rows >= B * Hq * Nq and last > 0, (ev, rows, last)   # every row, in each of its items
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=True, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), True, scale)
    assert_fwd(o, lse, ro, rl, f"planted decode, {splits} splits")


@pytest.mark.parametrize("scale", [0.05, 0.3, 1.0])
@pytest.mark.parametrize("d,causal", [(64, True), (128, False), (128, True)])
def test_scale_away_from_inverse_sqrt_d(cuda_lib, scale, d, causal):
    B, Hq, Hkv, N = 2, 4, 2, 700
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=int(scale * 1000) + d + int(causal))
    o, lse, dq, dk, dv = fwd_bwd(q, k, v, do, causal, scale)
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale)
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, scale)
    what = f"scale={scale} d={d} causal={causal}"
    assert_fwd(o, lse, ro, rl, what)
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, what)


@pytest.mark.parametrize("scale,d,causal", [(0.05, 128, True), (0.3, 64, False), (1.0, 128, True)])
def test_scale_deterministic_backward(cuda_lib, scale, d, causal):
    B, Hq, Hkv, N = 1, 4, 2, 500
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=700 + d)
    o, lse, dq, dk, dv = fwd_bwd(q, k, v, do, causal, scale, deterministic=True)
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, scale)
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, f"deterministic scale={scale}")


@pytest.mark.parametrize("scale,d,causal,splits", [(0.05, 64, False, 3), (1.0, 128, True, 4), (0.3, 128, False, 2)])
def test_scale_key_splits(cuda_lib, scale, d, causal, splits):
    B, Hq, Hkv, N = 1, 4, 1, 900
    q, k, v, _ = gen(B, Hq, Hkv, N, N, d, seed=800 + splits)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale)
    assert_fwd(o, lse, ro, rl, f"splits={splits} scale={scale}")
