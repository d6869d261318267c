"""Seeded synthetic inputs shared by the parity tests, the benchmark and the smoke check.

This module holds random-number generation and bf16 rounding only; it contains
none of the attention arithmetic, so the CUDA path and the CPU oracle can both
be fed from it without sharing any of the method.

Recipe (one CPU ``torch.Generator`` per workload, seeded with the workload's
seed): draw, in the fixed order q, k, v, dO, an fp32 ``randn`` tensor of shape
``[B, H, N, d]`` (``H = Hq`` for q and dO, ``Hkv`` for k and v), multiply q and
k by ``sigma_qk`` (3 for the numerically stressed workload, else 1), and round
each to bf16 (round to nearest even).  The oracle reads these exact bf16
values upcast to fp64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask, score scale and input recipe."""

    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma_qk: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def fwd_flops(self) -> float:
        """Forward FLOP convention: 4*B*Hq*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def bwd_flops(self) -> float:
        """Backward FLOP convention: 2.5x the forward count."""
        return 2.5 * self.fwd_flops

    def as_dict(self) -> dict:
        return asdict(self)


# The five workloads of the attention hot path.  Each is named by what it is,
# with its sizes.
WORKLOADS = {
    "tiny_b1_h1_n128_d64": Workload("tiny_b1_h1_n128_d64", 1, 1, 1, 128, 64, False, 0),
    "causal_b4_h16_n2048_d128": Workload("causal_b4_h16_n2048_d128", 4, 16, 16, 2048, 128, True, 1),
    "gqa_causal_b2_hq32_hkv8_n8192_d128": Workload(
        "gqa_causal_b2_hq32_hkv8_n8192_d128", 2, 32, 8, 8192, 128, True, 2),
    "long_causal_b1_h16_n32768_d128": Workload(
        "long_causal_b1_h16_n32768_d128", 1, 16, 16, 32768, 128, True, 3),
    "stressed_b8_h32_n4096_d64": Workload(
        "stressed_b8_h32_n4096_d64", 8, 32, 32, 4096, 64, False, 4, sigma_qk=3.0),
}

# The workload the benchmark reports on: the largest causal shape (B=1,
# H=16, N=32768, d=128); the others are timed beside it in the same run.
BENCH_WORKLOAD = "long_causal_b1_h16_n32768_d128"


def make_qkvdo(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int,
               sigma_qk: float = 1.0):
    """Return (q, k, v, dO) as contiguous bf16 CPU tensors, drawn per the recipe above."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)

    def draw(h: int, sigma: float) -> torch.Tensor:
        x = torch.randn((B, h, N, d), dtype=torch.float32, generator=g)
        if sigma != 1.0:
            x = x * sigma
        return x.to(torch.bfloat16).contiguous()

    q = draw(Hq, sigma_qk)
    k = draw(Hkv, sigma_qk)
    v = draw(Hkv, 1.0)
    do = draw(Hq, 1.0)
    return q, k, v, do


def make_workload_inputs(w: Workload):
    return make_qkvdo(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.sigma_qk)


def to_f64(t: torch.Tensor):
    """Exact upcast of a bf16 tensor to a float64 numpy array (for the oracle)."""
    return t.to(torch.float64).numpy()
