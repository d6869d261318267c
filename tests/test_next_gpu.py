"""GPU parity of the widened forward / backward (through the C ABI) against the
fp64 oracle: sliding window, key splits with the (O, LSE) merge, and decode
shapes (few queries against a long key/value history, grouped heads packed
into one tile)."""
import numpy as np
import pytest
import torch

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300.inputs import make_qkvdo
from oracle import ref
from tests.parity import assert_bwd, assert_fwd

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def f64(t):
    return t.double().numpy()


def gen(B, Hq, Hkv, Nq, Nk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Nq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Nk, d), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("N,d,window", [(300, 64, 1), (300, 128, 50), (1000, 64, 128), (1000, 128, 200),
                                        (700, 128, 129), (513, 64, 700)])
def test_window_forward_backward(cuda_lib, N, d, window):
    B, Hq, Hkv = 1, 4, 2
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=N + window)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward_ex(qd, kd, vd, causal=True, scale=scale, window=window)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=True, scale=scale, window=window)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), True, scale, window=window)
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), True, scale, window=window)
    assert_fwd(o, lse, ro, rl, f"window {window}")
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, f"window {window}")


@pytest.mark.parametrize("causal,window,splits", [(False, 0, 2), (True, 0, 3), (True, 0, 7), (False, 0, 16),
                                                  (True, 300, 4)])
def test_key_splits_merge(cuda_lib, causal, window, splits):
    B, Hq, Hkv, N, d = 2, 4, 1, 1100, 128
    q, k, v = gen(B, Hq, Hkv, N, N, d, seed=splits * 10 + int(causal))
    scale = d ** -0.5
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, window=window, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale, window=window)
    assert_fwd(o, lse, ro, rl, f"splits {splits}")


@pytest.mark.parametrize("Hq,Hkv,Nq,Nk,d,causal,splits", [
    (8, 2, 1, 4096, 128, True, 0),      # one new token, grouped heads packed into one tile
    (8, 2, 3, 1000, 64, True, 5),
    (32, 8, 1, 8192, 128, False, 0),
    (4, 4, 16, 2000, 128, True, 0),     # no grouping: per-head tiles of 16 rows
    (16, 1, 8, 700, 64, True, 2),       # multi-query: 16 heads x 8 rows fill one tile
    (8, 2, 100, 900, 128, True, 1),     # 4 x 100 rows do not fit one tile: per-head tiles
])
def test_decode_shapes(cuda_lib, Hq, Hkv, Nq, Nk, d, causal, splits):
    B = 2
    q, k, v = gen(B, Hq, Hkv, Nq, Nk, d, seed=Nq * 31 + Nk)
    scale = d ** -0.5
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), causal, scale)
    assert_fwd(o, lse, ro, rl, f"decode Nq={Nq} Nk={Nk}")


def test_decode_equals_last_rows_of_full_attention(cuda_lib):
    # The queries stand at the last Nq positions: the decode result equals the
    # last rows of causal self-attention over the whole sequence.
    B, Hq, Hkv, N, d, Nq = 1, 8, 2, 1024, 128, 5
    q, k, v = gen(B, Hq, Hkv, N, N, d, seed=77)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    of, lf = fa.forward(qd, kd, vd, causal=True)
    od, ld = fa.forward_ex(qd[:, :, N - Nq:].contiguous(), kd, vd, causal=True, num_splits=0)
    torch.cuda.synchronize()
    assert (od.float() - of[:, :, N - Nq:].float()).abs().max() <= 2e-2
    assert (ld - lf[:, :, N - Nq:]).abs().max() <= 1e-4 * max(1.0, lf.abs().max().item())


def test_splits_agree_with_one_pass(cuda_lib):
    B, Hq, Hkv, N, d = 1, 8, 8, 2048, 64
    q, k, v = gen(B, Hq, Hkv, N, N, d, seed=5)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o1, l1 = fa.forward_ex(qd, kd, vd, causal=True, num_splits=1)
    o4, l4 = fa.forward_ex(qd, kd, vd, causal=True, num_splits=4)
    torch.cuda.synchronize()
    assert (o1.float() - o4.float()).abs().max() <= 1e-2
    assert (l1 - l4).abs().max() <= 1e-4 * max(1.0, l1.abs().max().item())


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,window", [
    (1, 2, 1, 300, 64, True, 0),
    (2, 4, 2, 1000, 128, True, 0),
    (1, 4, 4, 513, 128, False, 0),
    (1, 2, 2, 700, 64, True, 150),
    (1, 8, 2, 129, 128, True, 1),
    # More query tiles than SMs: each persistent dQ CTA walks several items.
    (4, 12, 4, 1000, 128, True, 0),
    (4, 12, 12, 1000, 64, False, 0),
    (3, 8, 2, 1100, 128, True, 200),
])
def test_deterministic_backward(cuda_lib, B, Hq, Hkv, N, d, causal, window):
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=N * 3 + d + window)
    scale = d ** -0.5
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward_ex(qd, kd, vd, causal=causal, scale=scale, window=window)
    g1 = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, window=window, deterministic=True)
    g2 = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, window=window, deterministic=True)
    torch.cuda.synchronize()
    fa.check_device_status()
    # Bitwise reproducible, dQ included.
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), causal, scale, window=window)
    assert_bwd(*g1, rdq, rdk, rdv, f"deterministic N={N} window={window}")
    # Same dK, dV as the reduce-add backward (identical MMAs); dQ within rounding.
    g3 = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g3[1]) and torch.equal(g1[2], g3[2])
    assert (g1[0].float() - g3[0].float()).abs().max() <= 2e-2


def test_deterministic_backward_standard_workload(cuda_lib):
    from exact_io_aware_flashattention_gb300.inputs import WORKLOADS, make_workload_inputs
    w = WORKLOADS["causal_b4_h16_n2048_d128"]
    q, k, v, do = make_workload_inputs(w)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=True, scale=w.scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale, deterministic=True)
    torch.cuda.synchronize()
    fa.check_device_status()
    rdq, rdk, rdv = ref.attention_backward(f64(q), f64(k), f64(v), f64(do), True, w.scale)
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, "deterministic standard causal workload")


def test_more_splits_than_key_tiles(cuda_lib):
    # num_splits larger than the number of key tiles: every split holds at
    # least one tile (the chunk size is rounded up).
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 3, 300, 64
    q, k, v = gen(B, Hq, Hkv, Nq, Nk, d, seed=91)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=True, num_splits=100)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), True, d ** -0.5)
    assert_fwd(o, lse, ro, rl, "100 splits over 3 key tiles")


@pytest.mark.parametrize("N,window,splits", [(16, 0, 1), (16, 5, 1), (40, 0, 3), (130, 64, 2)])
def test_self_attention_through_fwd_ex(cuda_lib, N, window, splits):
    # Nq == Nk through the general entry point, with grouped heads small
    # enough to be packed into one tile (N = 16, 40) or not (N = 130).
    B, Hq, Hkv, d = 2, 8, 2, 128
    q, k, v = gen(B, Hq, Hkv, N, N, d, seed=N + window)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=True, window=window, num_splits=splits)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rl = ref.attention_forward(f64(q), f64(k), f64(v), True, d ** -0.5, window=window)
    assert_fwd(o, lse, ro, rl, f"N={N} window={window} splits={splits}")


def test_decode_grouped_at_scale(cuda_lib):
    # Grouped decode at the size of the grouped-query workload (32 query
    # heads over 8 kv heads, 8192 keys), 4 new rows per head, default splits;
    # the oracle checks two (batch, kv group) units drawn by seed.
    B, Hq, Hkv, Nq, Nk, d = 2, 32, 8, 4, 8192, 128
    q, k, v = gen(B, Hq, Hkv, Nq, Nk, d, seed=2024)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward_ex(qd, kd, vd, causal=True, num_splits=0)
    torch.cuda.synchronize()
    fa.check_device_status()
    G = Hq // Hkv
    rng = np.random.default_rng(7)
    for u in rng.choice(B * Hkv, size=2, replace=False):
        b, g = divmod(int(u), Hkv)
        hs = slice(g * G, (g + 1) * G)
        ro, rl = ref.attention_forward(f64(q[b:b + 1, hs]), f64(k[b:b + 1, g:g + 1]), f64(v[b:b + 1, g:g + 1]), True,
                                       d ** -0.5)
        assert_fwd(o[b:b + 1, hs], lse[b:b + 1, hs], ro, rl, f"decode unit (b={b}, kv={g})")
