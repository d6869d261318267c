"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle,
element by element, on seeded inputs.

* the tiny and the standard causal workload in full (the latter is the shape
  the benchmark times, in the same launch configuration);
* the GQA, long-context and stressed workloads at full size on the GPU, with
  the oracle on (batch, kv-group) units drawn by seed, plus properties that
  hold for every head;
* ragged and degenerate shapes: N in {1, 17, 127, 129, 200, 1000}, both head
  dims, causal and not, grouped heads.
"""
import numpy as np
import pytest
import torch

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300.inputs import WORKLOADS, make_qkvdo, make_workload_inputs, to_f64
from oracle import ref
from tests.parity import assert_bwd, assert_fwd, as_f64

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_gpu(q, k, v, do, causal, scale):
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    return o, lse, dq, dk, dv


def oracle(q, k, v, do, causal, scale):
    args = (to_f64(q), to_f64(k), to_f64(v))
    ro, rlse = ref.attention_forward(*args, causal, scale)
    rdq, rdk, rdv = ref.attention_backward(*args, to_f64(do), causal, scale)
    return ro, rlse, rdq, rdk, rdv


@pytest.mark.parametrize("name", ["tiny_b1_h1_n128_d64", "causal_b4_h16_n2048_d128"])
def test_workload_full_parity(cuda_lib, name):
    w = WORKLOADS[name]
    q, k, v, do = make_workload_inputs(w)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, w.causal, w.scale)
    ro, rlse, rdq, rdk, rdv = oracle(q, k, v, do, w.causal, w.scale)
    e = assert_fwd(o, lse, ro, rlse, name)
    g = assert_bwd(dq, dk, dv, rdq, rdk, rdv, name)
    print(name, e, g)


SAMPLED = {
    "gqa_causal_b2_hq32_hkv8_n8192_d128": 2,
    "long_causal_b1_h16_n32768_d128": 1,
    # Peaked rows (q, k ~ N(0, 9)): where the rounding of a dominant weight
    # shows, so more of its heads are checked.
    "stressed_b8_h32_n4096_d64": 16,
}


@pytest.mark.parametrize("name", sorted(SAMPLED))
def test_workload_sampled_parity(cuda_lib, name):
    w = WORKLOADS[name]
    q, k, v, do = make_workload_inputs(w)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, w.causal, w.scale)
    G = w.Hq // w.Hkv
    # Properties of every head: finite, and each O row is a convex combination
    # of V rows, so |O| <= max |V| of its kv head.
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    vmax = v.float().abs().amax(dim=(2, 3)).to(DEV)                      # [B, Hkv]
    omax = o.float().abs().amax(dim=(2, 3)).view(w.B, w.Hkv, G).amax(2)  # [B, Hkv]
    assert bool((omax <= vmax * (1 + 1e-2) + 1e-3).all())
    # Oracle on (batch, kv-group) units drawn by seed.
    rng = np.random.default_rng(1000 + w.seed)
    units = rng.choice(w.B * w.Hkv, size=SAMPLED[name], replace=False)
    for u in units:
        b, g = divmod(int(u), w.Hkv)
        hs = slice(g * G, (g + 1) * G)
        sub = (q[b:b + 1, hs], k[b:b + 1, g:g + 1], v[b:b + 1, g:g + 1], do[b:b + 1, hs])
        ro, rlse, rdq, rdk, rdv = oracle(*sub, w.causal, w.scale)
        what = f"{name} unit (b={b}, kv={g})"
        e = assert_fwd(o[b:b + 1, hs], lse[b:b + 1, hs], ro, rlse, what)
        gr = assert_bwd(dq[b:b + 1, hs], dk[b:b + 1, g:g + 1], dv[b:b + 1, g:g + 1], rdq, rdk, rdv, what)
        print(what, e, gr)


def test_stressed_forward_every_head(cuda_lib):
    """The stressed workload's forward on all 256 heads against the oracle.
    Its rows are peaked (q, k ~ N(0, 9)), where the bf16 rounding of a row's
    dominant weight shows in O; a CPU emulation of the kernel's arithmetic
    without the per-tile correction for it put 4 of 24 sampled heads above
    the 2e-2 max-abs bound, with it all below 0.016."""
    w = WORKLOADS["stressed_b8_h32_n4096_d64"]
    q, k, v, do = make_workload_inputs(w)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    o, lse = fa.forward(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    fa.check_device_status()
    ro, rlse = ref.attention_forward(to_f64(q), to_f64(k), to_f64(v), w.causal, w.scale)
    e = assert_fwd(o, lse, ro, rlse, "stressed workload, every head")
    print("stressed every head", e)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 127, 129, 200, 1000])
def test_ragged_shapes(cuda_lib, N, d, causal):
    B, Hq, Hkv = 1, 2, 1
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=N * 7 + d + int(causal))
    scale = 1.0 / np.sqrt(d)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, causal, scale)
    ro, rlse, rdq, rdk, rdv = oracle(q, k, v, do, causal, scale)
    assert_fwd(o, lse, ro, rlse, f"N={N} d={d} causal={causal}")
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (3, 4, 4, 384, 128, True),     # multi-head, several batches
    (2, 4, 1, 300, 64, True),      # multi-query
    (1, 8, 2, 512, 128, False),    # grouped
    (2, 6, 3, 257, 64, False),
])
def test_head_groupings(cuda_lib, B, Hq, Hkv, N, d, causal):
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=B * 100 + Hq * 10 + Hkv)
    scale = 1.0 / np.sqrt(d)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, causal, scale)
    ro, rlse, rdq, rdk, rdv = oracle(q, k, v, do, causal, scale)
    assert_fwd(o, lse, ro, rlse)
    assert_bwd(dq, dk, dv, rdq, rdk, rdv)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_many_items_per_cta_ragged(cuda_lib, d, causal):
    """More (query tile, head) items than SMs with a ragged last tile, so every
    persistent CTA finishes several items whose O goes out through the Q slot
    it is staged in, partial tiles included, and each dK/dV CTA walks several
    units."""
    B, Hq, Hkv, N = 4, 12, 12, 1000
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=4000 + d)
    scale = 1.0 / np.sqrt(d)
    o, lse, dq, dk, dv = run_gpu(q, k, v, do, causal, scale)
    ro, rlse, rdq, rdk, rdv = oracle(q, k, v, do, causal, scale)
    assert_fwd(o, lse, ro, rlse, f"many items d={d} causal={causal}")
    assert_bwd(dq, dk, dv, rdq, rdk, rdv, f"many items d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_dkdv_outputs_only_16_byte_aligned(cuda_lib, d):
    """dK / dV at addresses that are 16- but not 32-byte aligned (allowed by
    the ABI) take the 16-byte store path and give the same bits."""
    B, Hq, Hkv, N = 2, 4, 2, 384
    q, k, v, do = (t.to(DEV) for t in make_qkvdo(B, Hq, Hkv, N, d, seed=77 + d))
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    _, dk_ref, dv_ref = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    n = k.numel()
    buf = torch.empty(2 * n + 64, dtype=torch.bfloat16, device=DEV)
    assert buf.data_ptr() % 32 == 0
    dk = buf[8:8 + n].view(k.shape)              # 16 bytes past a 32-byte boundary
    dv = buf[n + 40:2 * n + 40].view(v.shape)
    assert dk.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16
    fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, dk=dk, dv=dv)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_deterministic_dq_only_16_byte_aligned(cuda_lib, d):
    """The deterministic dQ kernel writes a 16- (not 32-) byte aligned dQ through
    its 16-byte store path, bit for bit as an aligned one."""
    B, Hq, Hkv, N = 2, 4, 2, 384
    q, k, v, do = (t.to(DEV) for t in make_qkvdo(B, Hq, Hkv, N, d, seed=99 + d))
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.forward(q, k, v, causal=True, scale=scale)
    dq_ref, _, _ = fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True)
    n = q.numel()
    buf = torch.empty(n + 32, dtype=torch.bfloat16, device=DEV)
    dq = buf[8:8 + n].view(q.shape)
    assert dq.data_ptr() % 32 == 16
    fa.backward(q, k, v, o, lse, do, causal=True, scale=scale, deterministic=True, dq=dq)
    torch.cuda.synchronize()
    fa.check_device_status()
    assert torch.equal(dq, dq_ref)


def test_gqa_equals_repeated_heads_on_gpu(cuda_lib):
    # Grouped attention == multi-head attention on K/V repeated per group.
    B, Hq, Hkv, N, d = 1, 8, 2, 640, 128
    q, k, v, do = make_qkvdo(B, Hq, Hkv, N, d, seed=5)
    rk, rv = (t.repeat_interleave(Hq // Hkv, dim=1).contiguous() for t in (k, v))
    o1, l1, dq1, dk1, dv1 = run_gpu(q, k, v, do, True, d ** -0.5)
    o2, l2, dq2, dk2, dv2 = run_gpu(q, rk, rv, do, True, d ** -0.5)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    dk2 = dk2.float().view(B, Hkv, Hq // Hkv, N, d).sum(2)
    dv2 = dv2.float().view(B, Hkv, Hq // Hkv, N, d).sum(2)
    assert (dk1.float() - dk2).norm() / dk2.norm() < 1e-2
    assert (dv1.float() - dv2).norm() / dv2.norm() < 1e-2


def test_causal_row0_and_constant_v_on_gpu(cuda_lib):
    N, d = 300, 64
    q, k, v, do = make_qkvdo(1, 1, 1, N, d, seed=11)
    o, lse, *_ = run_gpu(q, k, v, do, True, 0.125)
    assert torch.equal(o[0, 0, 0].cpu(), v[0, 0, 0])               # row 0 sees only key 0
    s00 = 0.125 * float((q[0, 0, 0].double() * k[0, 0, 0].double()).sum())
    assert abs(float(lse[0, 0, 0]) - s00) <= 1e-4 * max(1.0, abs(s00))
    vc = v[:, :, :1].expand_as(v).contiguous()
    o, _, dq, dk, _ = run_gpu(q, k, vc, do, False, 0.125)
    assert (o.float().cpu() - vc.float()).abs().max() <= 1e-2
    assert dq.float().abs().max() <= 2e-2 and dk.float().abs().max() <= 2e-2


def test_dkdv_deterministic(cuda_lib):
    q, k, v, do = make_qkvdo(1, 4, 2, 1024, 128, seed=12)
    r1 = run_gpu(q, k, v, do, True, 0.088)
    r2 = run_gpu(q, k, v, do, True, 0.088)
    assert torch.equal(r1[0], r2[0]) and torch.equal(r1[1], r2[1])
    assert torch.equal(r1[3], r2[3]) and torch.equal(r1[4], r2[4])
    assert (r1[2].float() - r2[2].float()).abs().max() <= 1e-2


def test_long_context_memory_is_linear(cuda_lib):
    # No N x N buffer: the library allocates nothing, and the only scratch is
    # the O(N d) workspace.  Free device memory must not drop during the calls.
    w = WORKLOADS["long_causal_b1_h16_n32768_d128"]
    q, k, v, do = (t.to(DEV) for t in make_workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=DEV)
    ws = fa.workspace_for(w.B, w.Hq, w.Hkv, w.N, w.d, DEV)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    fa.backward(q, k, v, o, lse, do, causal=True, scale=w.scale, workspace=ws, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free0 - free1 < 64 * 2 ** 20
    assert ws.numel() < 300 * 2 ** 20                      # vs 68.7 GB for fp32 S of 16 heads
    fa.check_device_status()


def test_bounded_wait_reports_timeout_and_device_survives(cuda_lib):
    assert fa.fa_selftest_wait_timeout(2_000_000) == fa.FA_OK
    status, detail = fa.fa_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert status == fa.FA_ERR_DEVICE_TIMEOUT
    assert detail[1] == 99
    status, _ = fa.fa_last_device_status(torch.cuda.current_stream().cuda_stream)
    assert status == fa.FA_OK
    # The context is still usable.
    q, k, v, do = make_qkvdo(1, 1, 1, 128, 64, seed=0)
    o, lse, *_ = run_gpu(q, k, v, do, False, 0.125)
    ro, rlse = ref.attention_forward(to_f64(q), to_f64(k), to_f64(v), False, 0.125)
    assert_fwd(o, lse, ro, rlse)


def test_failed_drain_refuses_further_launches(cuda_lib):
    """A drain wait that gives up (the self-test's barrier is never completed;
    nothing is in flight and nothing faults) is reported as
    FA_ERR_DEVICE_DRAIN, after which the library refuses every launch on the
    device.  That state lasts for the process, so it runs in a child."""
    import os
    import subprocess
    import sys
    import textwrap
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent("""
        import torch
        import exact_io_aware_flashattention_gb300 as fa
        fa.load_library()
        s = torch.cuda.current_stream().cuda_stream
        q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
        args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 1, 128, 64, 0, 0.125, s)
        assert fa.fa_fwd(*args) == fa.FA_OK
        assert fa.fa_last_device_status(s)[0] == fa.FA_OK
        assert fa.fa_selftest_drain_timeout(2_000_000, s) == fa.FA_OK
        st, detail = fa.fa_last_device_status(s)
        assert st == fa.FA_ERR_DEVICE_DRAIN and detail[1] == 98, (st, detail)
        assert fa.fa_fwd(*args) == fa.FA_ERR_DEVICE_DRAIN
        assert fa.fa_selftest_wait_timeout(2_000_000, s) == fa.FA_ERR_DEVICE_DRAIN
        assert fa.fa_last_device_status(s)[0] == fa.FA_ERR_DEVICE_DRAIN
        torch.cuda.synchronize()          # the CUDA context itself is fine
        print("drain refusal ok")
    """)
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "drain refusal ok" in r.stdout, r.stdout + r.stderr
