"""Host-side checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/fa.h declares, and invalid arguments are
rejected with the documented status before any CUDA call."""
import ctypes

import pytest

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def test_header_declares_the_boundary():
    names = fa.header_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_strerror", "fa_last_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in fa.header_functions():
        assert hasattr(lib, name), f"{name} declared in include/fa.h but not exported"


def test_binding_exposes_same_names():
    for name in fa.header_functions():
        assert callable(getattr(fa, name, None)), f"binding lacks {name}"


def test_version_and_strerror(lib):
    assert fa.fa_version() == 101
    for code in range(0, 14):
        assert fa.fa_strerror(code) and fa.fa_strerror(code) != "unknown status"
    assert "no further launches" in fa.fa_strerror(fa.FA_ERR_DEVICE_DRAIN)
    assert fa.fa_strerror(999) == "unknown status"


def test_workspace_formula_is_linear_in_n(lib):
    # dQ accumulator fp32 [B,Hq,N,d] + LSE*log2e and D, fp32 [B*Hq, ceil(N/128)*128]
    # each; every part rounded up to 256 B.
    def expect(B, Hq, N, d):
        r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
        ntp = (N + 127) // 128 * 128
        return r256(B * Hq * N * d * 4) + 2 * r256(B * Hq * ntp * 4)
    for shape in [(1, 1, 1, 128, 64), (4, 16, 16, 2048, 128), (1, 16, 16, 32768, 128), (2, 32, 8, 8192, 128)]:
        B, Hq, Hkv, N, d = shape
        assert fa.fa_bwd_workspace_bytes(B, Hq, Hkv, N, d) == expect(B, Hq, N, d)
    # O(N): doubling N doubles it (up to rounding), never N^2.
    w1 = fa.fa_bwd_workspace_bytes(1, 16, 16, 16384, 128)
    w2 = fa.fa_bwd_workspace_bytes(1, 16, 16, 32768, 128)
    assert abs(w2 - 2 * w1) <= 512
    # The N x N fp32 buffer the long-context shape avoids: 16 * 32768^2 * 4 B = 68.7 GB.
    assert w2 < 16 * 32768 ** 2 * 4 / 200
    assert fa.fa_bwd_workspace_bytes(1, 3, 2, 128, 128) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 128, 96) == 0


A = 1 << 20  # fake, 16-byte aligned, non-overlapping "device" addresses (never dereferenced)


def _fwd(**kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, Hq=1, Hkv=1, N=16, d=64, causal=0,
                scale=0.125, stream=None)
    args.update(kw)
    return fa.fa_fwd(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), fa.FA_ERR_NULL_PTR),
    (dict(lse=None), fa.FA_ERR_NULL_PTR),
    (dict(B=0), fa.FA_ERR_BAD_SHAPE),
    (dict(N=0), fa.FA_ERR_BAD_SHAPE),
    (dict(Hq=3, Hkv=2), fa.FA_ERR_BAD_SHAPE),
    (dict(B=70000), fa.FA_ERR_BAD_SHAPE),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED_HEADDIM),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED_HEADDIM),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(scale=0.0), fa.FA_ERR_BAD_ARGUMENT),
    (dict(scale=float("nan")), fa.FA_ERR_BAD_ARGUMENT),
    (dict(scale=-1.0), fa.FA_ERR_BAD_ARGUMENT),
    (dict(causal=2), fa.FA_ERR_BAD_ARGUMENT),
    (dict(o=A + 256), fa.FA_ERR_ALIASING),
])
def test_fwd_rejects_bad_arguments(lib, kw, status):
    assert _fwd(**kw) == status


def test_bwd_rejects_bad_arguments(lib):
    ws = fa.fa_bwd_workspace_bytes(1, 2, 1, 64, 128)
    base = dict(q=A, k=2 * A, v=3 * A, o=4 * A, do=5 * A, lse=6 * A, dq=7 * A, dk=8 * A, dv=9 * A,
                B=1, Hq=2, Hkv=1, N=64, d=128, causal=1, scale=0.088, workspace=10 * A,
                workspace_bytes=ws, stream=None)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return fa.fa_bwd(**a)
    assert call(workspace_bytes=ws - 1) == fa.FA_ERR_WORKSPACE_TOO_SMALL
    assert call(workspace=None) == fa.FA_ERR_NULL_PTR
    assert call(dq=A) == fa.FA_ERR_ALIASING
    assert call(dk=A + 16) == fa.FA_ERR_ALIASING
    assert call(Hkv=4) == fa.FA_ERR_BAD_SHAPE
    assert call(d=32) == fa.FA_ERR_UNSUPPORTED_HEADDIM
    assert call(dv=9 * A + 4) == fa.FA_ERR_MISALIGNED
    assert fa.fa_bwd_dq_convert(None, 1, 2, 1, 64, 128, 0.1, 10 * A, ws, None) == fa.FA_ERR_NULL_PTR
    assert fa.fa_bwd_preprocess(4 * A, 5 * A, 6 * A, 1, 2, 1, 64, 128, 10 * A, 16, None) == \
        fa.FA_ERR_WORKSPACE_TOO_SMALL
    assert fa.fa_bwd_preprocess(4 * A, 5 * A, None, 1, 2, 1, 64, 128, 10 * A, ws, None) == fa.FA_ERR_NULL_PTR
    assert call(lse=None) == fa.FA_ERR_NULL_PTR
    assert call(lse=6 * A + 8) == fa.FA_ERR_MISALIGNED


def test_selftest_rejects_bad_limit(lib):
    assert fa.fa_selftest_wait_timeout(10) == fa.FA_ERR_BAD_ARGUMENT


def _fwd_ex(**kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, Hq=2, Hkv=1, Nq=4, Nk=300, d=64, causal=1, window=0,
                num_splits=1, scale=0.125, workspace=None, workspace_bytes=0, stream=None)
    args.update(kw)
    return fa.fa_fwd_ex(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(window=-1), fa.FA_ERR_BAD_ARGUMENT),
    (dict(window=4, causal=0), fa.FA_ERR_BAD_ARGUMENT),
    (dict(Nq=400), fa.FA_ERR_BAD_ARGUMENT),          # causal with more queries than keys
    (dict(num_splits=0), fa.FA_ERR_BAD_ARGUMENT),
    (dict(Nk=0), fa.FA_ERR_BAD_SHAPE),
    (dict(num_splits=2), fa.FA_ERR_NULL_PTR),        # splits need a workspace
    (dict(num_splits=2, workspace=6 * A, workspace_bytes=64), fa.FA_ERR_WORKSPACE_TOO_SMALL),
    (dict(num_splits=2, workspace=6 * A + 4, workspace_bytes=1 << 20), fa.FA_ERR_MISALIGNED),
    (dict(num_splits=2, workspace=A, workspace_bytes=1 << 20), fa.FA_ERR_ALIASING),
])
def test_fwd_ex_rejects_bad_arguments(lib, kw, status):
    assert _fwd_ex(**kw) == status


def test_fwd_ex_workspace_formula(lib):
    # Per-split O fp32 [S, B*Hq*Nq, d] then per-split LSE fp32 [S, B*Hq*Nq], 256-B aligned parts.
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for B, Hq, Hkv, Nq, Nk, d, S in [(1, 8, 2, 1, 8192, 128, 8), (4, 32, 8, 3, 32768, 64, 16), (2, 2, 2, 100, 300, 64, 3)]:
        rows = B * Hq * Nq
        assert fa.fa_fwd_ex_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, S) == r256(S * rows * d * 4) + r256(S * rows * 4)
    assert fa.fa_fwd_ex_workspace_bytes(1, 8, 2, 1, 8192, 128, 1) == 0
    assert fa.fa_fwd_ex_workspace_bytes(1, 8, 3, 1, 8192, 128, 4) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(window=-1), fa.FA_ERR_BAD_ARGUMENT),
    (dict(window=8, causal=0), fa.FA_ERR_BAD_ARGUMENT),
    (dict(deterministic=2), fa.FA_ERR_BAD_ARGUMENT),
])
def test_bwd_ex_rejects_bad_window(lib, kw, status):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, do=5 * A, lse=6 * A, dq=7 * A, dk=8 * A, dv=9 * A, B=1, Hq=1, Hkv=1,
                N=16, d=64, causal=1, window=0, deterministic=0, scale=0.125, workspace=10 * A, workspace_bytes=1 << 20,
                stream=None)
    args.update(kw)
    assert fa.fa_bwd_ex(**args) == status
