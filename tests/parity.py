"""Parity metrics and tolerances for comparing the CUDA path with the CPU oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs):
  O    : max-abs <= 2e-2 and relative L2 <= 5e-3
  LSE  : max_i |LSE_i - ref_i| / max(1, |ref_i|) <= 1e-4
  dQ, dK, dV : relative L2 <= 1e-2
relative L2 = ||x - ref||_2 / ||ref||_2 over the whole tensor.
"""
import numpy as np

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_REL = 1e-4
GRAD_REL_L2 = 1e-2


def as_f64(t):
    return t.detach().float().cpu().double().numpy()


def rel_l2(x, ref):
    den = np.linalg.norm(ref)
    if den == 0:
        return float(np.linalg.norm(x))
    return float(np.linalg.norm(x - ref) / den)


def fwd_errors(o, lse, ro, rlse):
    o = as_f64(o) if not isinstance(o, np.ndarray) else o
    lse = as_f64(lse) if not isinstance(lse, np.ndarray) else lse
    return {
        "o_max_abs": float(np.abs(o - ro).max()),
        "o_rel_l2": rel_l2(o, ro),
        "lse_rel": float((np.abs(lse - rlse) / np.maximum(1.0, np.abs(rlse))).max()),
    }


def assert_fwd(o, lse, ro, rlse, what=""):
    e = fwd_errors(o, lse, ro, rlse)
    assert np.all(np.isfinite(as_f64(o) if not isinstance(o, np.ndarray) else o)), f"{what}: non-finite O"
    assert e["o_max_abs"] <= O_MAX_ABS, f"{what}: O max-abs {e}"
    assert e["o_rel_l2"] <= O_REL_L2, f"{what}: O rel-L2 {e}"
    assert e["lse_rel"] <= LSE_REL, f"{what}: LSE {e}"
    return e


def assert_bwd(dq, dk, dv, rdq, rdk, rdv, what=""):
    errs = {}
    for name, g, r in (("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        g = as_f64(g) if not isinstance(g, np.ndarray) else g
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        errs[name] = rel_l2(g, r)
        assert errs[name] <= GRAD_REL_L2, f"{what}: {name} rel-L2 {errs}"
    return errs


class GuardedBuffers:
    """Output buffers with guard bytes on both sides.

    ``empty(shape, dtype)`` returns a contiguous CUDA view into a larger byte
    buffer whose first and last GUARD bytes (and the view itself) are filled
    with a fixed pattern; ``check()`` asserts that no guard byte changed, i.e.
    that no kernel wrote outside the output it was given.  The views start
    GUARD bytes into a fresh allocation, so they keep its 256-byte alignment.
    """

    GUARD = 4096
    PATTERN = 0xA5

    def __init__(self, device):
        self.device = device
        self.bufs = []

    def empty(self, shape, dtype):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((n + 2 * self.GUARD,), self.PATTERN, dtype=torch.uint8, device=self.device)
        self.bufs.append((raw, n))
        return raw[self.GUARD:self.GUARD + n].view(dtype).view(*shape)

    def check(self):
        for raw, n in self.bufs:
            head = raw[:self.GUARD]
            tail = raw[self.GUARD + n:]
            assert bool((head == self.PATTERN).all()), "guard bytes before an output were overwritten"
            assert bool((tail == self.PATTERN).all()), "guard bytes after an output were overwritten"
