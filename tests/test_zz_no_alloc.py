"""fa_bwd_noalloc, the backward pass for callers that cannot allocate device
memory (for example code running under a memory manager that owns the whole
device, or a plugin host that forbids cudaMalloc at run time).  Its scratch is
a fixed buffer compiled into the library, so it takes no workspace argument.

Checked through the C ABI on two calls in a row with different problems (the
second call also shows that what the first call left in the shared buffer
does not leak into its result): against the fp64 CPU oracle at the parity
tolerance, and against fa_bwd with a caller-owned workspace.  The second
problem uses a softmax scale away from 1/sqrt(d).  This file is collected
last so that a run stopping at the first failure has already run every other
test.
"""
import pytest
import torch

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300.inputs import make_qkvdo, to_f64
from oracle import ref
from tests.parity import GRAD_REL_L2, as_f64, assert_bwd, rel_l2

pytestmark = pytest.mark.gpu

PROBLEMS = [
    # B, Hq, Hkv, N, d, causal, scale, seed
    (2, 4, 2, 1000, 128, True, 128 ** -0.5, 77),
    (1, 6, 3, 777, 64, False, 0.3, 78),
]


def _run_pair(B, Hq, Hkv, N, d, causal, scale, seed):
    assert fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d) <= fa.NOALLOC_SCRATCH_BYTES
    qh, kh, vh, doh = make_qkvdo(B, Hq, Hkv, N, d, seed=seed)
    q, k, v, do = (t.cuda() for t in (qh, kh, vh, doh))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    want = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale)   # existing entry point
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()
    allocated = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    status = fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                               lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                               B, Hq, Hkv, N, d, causal, scale, torch.cuda.current_stream().cuda_stream)
    assert status == fa.FA_OK, fa.fa_strerror(status)
    torch.cuda.synchronize()
    fa.check_device_status()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == allocated
    assert free_before - free_after < 2 * 2 ** 20
    rdq, rdk, rdv = ref.attention_backward(to_f64(qh), to_f64(kh), to_f64(vh), to_f64(doh), causal, scale)
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, f"fa_bwd_noalloc vs oracle, N={N} d={d} scale={scale:.3g}")
    for name, got, other in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        err = rel_l2(as_f64(got), as_f64(other))
        assert err <= GRAD_REL_L2, f"{name}: rel-L2 {err} vs fa_bwd"


def test_noalloc_backward_matches_oracle_and_fa_bwd_on_two_calls(cuda_lib):
    for problem in PROBLEMS:
        _run_pair(*problem)


def test_noalloc_rejects_problems_beyond_its_buffer(cuda_lib):
    # 2 * 16 * 4096 * 129 * 4 bytes of scratch > 32 MiB: refused before any launch.
    B, Hq, Hkv, N, d = 2, 16, 16, 4096, 128
    assert fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d) > fa.NOALLOC_SCRATCH_BYTES
    status = fa.fa_bwd_noalloc(16, 32, 48, 64, 80, 96, 112, 128, 144, B, Hq, Hkv, N, d, 1, 0.088,
                               torch.cuda.current_stream().cuda_stream)
    assert status == fa.FA_ERR_SCRATCH_LIMIT
    assert "FA_NOALLOC_SCRATCH_BYTES" in fa.fa_strerror(status)
