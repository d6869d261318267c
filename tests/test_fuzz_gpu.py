"""Seeded random sweep of the CUDA path against the oracle.

Each case draws, from one fixed seed: batch, kv heads and group size (GQA),
query and key lengths (ragged, from 1 up to several tiles; fewer queries than
keys for the decode-shaped forward, queries at the last positions), head dim
64 or 128, causal or not, a sliding window (causal only), the number of key
splits of the forward (1-6, more than the key tiles at small N), the softmax scale (1/sqrt(d) or an arbitrary value),
the spread of q and k, and the deterministic or reduce-add backward.  Outputs
live between guard bytes, so a write outside any output fails the case.

The cases complement the hand-picked ones in the other GPU files: they cross
features (e.g. a window with key splits at d = 64 and a group of 4) that no
single parity test combines.
"""
import math

import numpy as np
import pytest
import torch

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300.inputs import make_qkvdo, to_f64
from oracle import ref
from tests.parity import GRAD_REL_L2, GuardedBuffers, as_f64, assert_bwd, assert_fwd, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
N_CASES = 96


def draw_cases(n=N_CASES, seed=20261203):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        d = int(rng.choice([64, 128]))
        B = int(rng.integers(1, 4))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 4]))
        Nk = int(rng.choice([int(rng.integers(1, 130)), int(rng.integers(130, 700))]))
        decode = bool(rng.random() < 0.25)
        Nq = int(rng.integers(1, Nk + 1)) if decode else Nk
        causal = bool(rng.random() < 0.6)
        window = int(rng.integers(1, Nk + 1)) if causal and rng.random() < 0.4 else 0
        splits = int(rng.integers(1, 7))   # may exceed the key tiles: the library clamps
        scale = 1.0 / math.sqrt(d) if rng.random() < 0.5 else float(rng.uniform(0.02, 0.4))
        sigma = float(rng.choice([1.0, 2.0]))
        deterministic = bool(rng.random() < 0.4)
        # Keep the fp64 oracle to about a second per case.
        if B * Hkv * G * Nq * Nk * d > 4e8:
            continue
        cases.append(dict(B=B, Hkv=Hkv, Hq=Hkv * G, Nq=Nq, Nk=Nk, d=d, causal=causal, window=window,
                          splits=splits, scale=scale, sigma=sigma, deterministic=deterministic,
                          seed=int(rng.integers(0, 2**31 - 1))))
    return cases


CASES = draw_cases()


def case_id(c):
    return (f"B{c['B']}-hq{c['Hq']}-hkv{c['Hkv']}-nq{c['Nq']}-nk{c['Nk']}-d{c['d']}"
            f"-{'c' if c['causal'] else 'nc'}-w{c['window']}-s{c['splits']}-{'det' if c['deterministic'] else 'red'}")


def test_cases_cover_the_features():
    """The draw is fixed; this checks it still crosses the features it is meant to."""
    assert len(CASES) == N_CASES
    assert {c["d"] for c in CASES} == {64, 128}
    assert any(c["Hq"] > c["Hkv"] for c in CASES)
    assert any(c["Nq"] < c["Nk"] for c in CASES)
    assert any(c["window"] > 0 for c in CASES)
    assert any(c["splits"] > 1 for c in CASES)
    assert any(c["splits"] > -(-c["Nk"] // 128) for c in CASES)
    assert any(c["deterministic"] and c["Nq"] == c["Nk"] for c in CASES)
    assert any(c["Nk"] % 128 != 0 and c["Nk"] > 128 for c in CASES)
    assert any(abs(c["scale"] - 1.0 / math.sqrt(c["d"])) > 1e-3 for c in CASES)


@pytest.mark.parametrize("c", CASES, ids=[case_id(c) for c in CASES])
def test_fuzz_case(cuda_lib, c):
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    q, k, v, do = make_qkvdo(B, Hq, Hkv, Nk, d, c["seed"], sigma_qk=c["sigma"])
    q, do = q[:, :, Nk - Nq:].contiguous(), do[:, :, Nk - Nq:].contiguous()
    guards = GuardedBuffers(DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o = guards.empty((B, Hq, Nq, d), torch.bfloat16)
    lse = guards.empty((B, Hq, Nq), torch.float32)
    fa.forward_ex(qd, kd, vd, causal=c["causal"], scale=c["scale"], window=c["window"], num_splits=c["splits"],
                  out=o, lse=lse)
    grads = None
    if Nq == Nk:
        dq = guards.empty((B, Hq, Nq, d), torch.bfloat16)
        dk = guards.empty((B, Hkv, Nk, d), torch.bfloat16)
        dv = guards.empty((B, Hkv, Nk, d), torch.bfloat16)
        fa.backward(qd, kd, vd, o, lse, dod, causal=c["causal"], scale=c["scale"], window=c["window"],
                    deterministic=c["deterministic"], dq=dq, dk=dk, dv=dv)
        grads = (dq, dk, dv)
    torch.cuda.synchronize()
    fa.check_device_status()
    guards.check()

    args = (to_f64(q), to_f64(k), to_f64(v))
    ro, rlse = ref.attention_forward(*args, c["causal"], c["scale"], window=c["window"])
    what = case_id(c)
    assert_fwd(o, lse, ro, rlse, what)
    if grads is not None:
        rdq, rdk, rdv = ref.attention_backward(*args, to_f64(do), c["causal"], c["scale"], window=c["window"])
        # The backward works from the saved bf16 O: D = rowsum(dO * O) carries
        # O's rounding, which a row that sees few keys (dP - D cancels) turns
        # into a dQ / dK error of its own.  The oracle with D from its O rounded
        # to bf16 gives that floor; the CUDA path must match that reference
        # within the tolerance, and the exact one within tolerance + floor.
        ro_bf16 = torch.from_numpy(ro).to(torch.bfloat16).double().numpy()
        fdq, fdk, fdv = ref.attention_backward(*args, to_f64(do), c["causal"], c["scale"], window=c["window"],
                                               o_for_d=ro_bf16)
        assert_bwd(*grads, fdq, fdk, fdv, what + " (D from bf16 O)")
        for name, g, r, f in (("dq", grads[0], rdq, fdq), ("dk", grads[1], rdk, fdk), ("dv", grads[2], rdv, fdv)):
            floor = rel_l2(f, r)
            err = rel_l2(as_f64(g), r)
            assert err <= GRAD_REL_L2 + floor, f"{what}: {name} rel-L2 {err} against the exact oracle (floor {floor})"
