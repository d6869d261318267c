"""Thin Python binding of libfa_gb300.so (exact IO-aware attention on GB300).

The names ``fa_fwd``, ``fa_fwd_ex``, ``fa_fwd_ex_workspace_bytes``,
``fa_fwd_ex_default_splits``, ``fa_bwd``, ``fa_bwd_ex``, ``fa_bwd_preprocess``,
``fa_bwd_dkdv``, ``fa_bwd_dq_convert``, ``fa_bwd_workspace_bytes``, ``fa_strerror``,
``fa_last_device_status``, ``fa_selftest_wait_timeout``,
``fa_selftest_drain_timeout``, ``fa_bwd_noalloc``, ``fa_last_cuda_error`` and
``fa_version`` are
the C entry points of ``include/fa.h`` with the same arguments (pointers as
Python ints, stream as an int handle); they return the integer status.

``forward``/``backward`` marshal torch CUDA tensors into those calls: they
check dtype, shape, contiguity and device, allocate outputs with torch, pass
``data_ptr()`` and the current stream, and raise ``FAError`` on a non-zero
status.  Every step of the computation runs in the library's kernels; there
is no fallback of any kind.  If the library has not been built the first call
raises ``FAError``.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "_lib", "libfa_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(PKG_DIR), "include", "fa.h")

FA_OK = 0
FA_ERR_NULL_PTR = 1
FA_ERR_BAD_SHAPE = 2
FA_ERR_UNSUPPORTED_HEADDIM = 3
FA_ERR_MISALIGNED = 4
FA_ERR_WORKSPACE_TOO_SMALL = 5
FA_ERR_UNSUPPORTED_DEVICE = 6
FA_ERR_LAUNCH = 7
FA_ERR_DEVICE_TIMEOUT = 8
FA_ERR_CUDA = 9
FA_ERR_BAD_ARGUMENT = 10
FA_ERR_ALIASING = 11
FA_ERR_SCRATCH_LIMIT = 12
FA_ERR_DEVICE_DRAIN = 13
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class FAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({_strerror_safe(status)})" if what else
                         f"status {status} ({_strerror_safe(status)})")


_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "fa_fwd": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p], _i),
    "fa_fwd_ex": ([_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p], _i),
    "fa_fwd_ex_workspace_bytes": ([_i, _i, _i, _i, _i, _i, _i], _sz),
    "fa_fwd_ex_default_splits": ([_i, _i, _i, _i, _i, _i, _i, _i], _i),
    "fa_bwd_ex": ([_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p], _i),
    "fa_bwd_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "fa_bwd": ([_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p], _i),
    "fa_bwd_preprocess": ([_p, _p, _p, _i, _i, _i, _i, _i, _p, _sz, _p], _i),
    "fa_bwd_dkdv": ([_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p, _sz, _p], _i),
    "fa_bwd_dq_convert": ([_p, _i, _i, _i, _i, _i, _f, _p, _sz, _p], _i),
    "fa_strerror": ([_i], ctypes.c_char_p),
    "fa_last_device_status": ([_p, ctypes.POINTER(ctypes.c_int)], _i),
    "fa_selftest_wait_timeout": ([ctypes.c_ulonglong, _p], _i),
    "fa_selftest_drain_timeout": ([ctypes.c_ulonglong, _p], _i),
    "fa_version": ([], _i),
    "fa_last_cuda_error": ([], ctypes.c_char_p),
    "fa_bwd_noalloc": ([_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p], _i),
}


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle; raises FAError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FAError(FA_ERR_LAUNCH, f"CUDA library not built at {p} (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def header_functions(path: str = HEADER_PATH) -> list[str]:
    """Names of the functions include/fa.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\**\s*(fa_\w+)\s*\(", text, flags=re.M)))


def _strerror_safe(status: int) -> str:
    try:
        return load_library().fa_strerror(status).decode()
    except Exception:
        return "library not loaded"


# ---------------------------------------------------------------------------
# Raw entry points (same names and arguments as the C ABI).
# ---------------------------------------------------------------------------

def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, stream):
    return load_library().fa_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, int(causal), float(scale), stream)


def fa_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, window, num_splits, scale, workspace,
              workspace_bytes, stream):
    return load_library().fa_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, int(causal), int(window),
                                     int(num_splits), float(scale), workspace, workspace_bytes, stream)


def fa_fwd_ex_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits):
    return load_library().fa_fwd_ex_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits)


def fa_fwd_ex_default_splits(B, Hq, Hkv, Nq, Nk, d, causal, window):
    return load_library().fa_fwd_ex_default_splits(B, Hq, Hkv, Nq, Nk, d, int(causal), int(window))


def fa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, window, deterministic, scale, workspace,
              workspace_bytes, stream):
    return load_library().fa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), int(window),
                                    int(deterministic), float(scale), workspace, workspace_bytes, stream)


def fa_bwd_workspace_bytes(B, Hq, Hkv, N, d):
    return load_library().fa_bwd_workspace_bytes(B, Hq, Hkv, N, d)


def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, stream):
    return load_library().fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                                 workspace, workspace_bytes, stream)


def fa_bwd_preprocess(o, do, lse, B, Hq, Hkv, N, d, workspace, workspace_bytes, stream):
    return load_library().fa_bwd_preprocess(o, do, lse, B, Hq, Hkv, N, d, workspace, workspace_bytes, stream)


def fa_bwd_dkdv(q, k, v, do, dk, dv, B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, stream):
    return load_library().fa_bwd_dkdv(q, k, v, do, dk, dv, B, Hq, Hkv, N, d, int(causal), float(scale),
                                      workspace, workspace_bytes, stream)


def fa_bwd_dq_convert(dq, B, Hq, Hkv, N, d, scale, workspace, workspace_bytes, stream):
    return load_library().fa_bwd_dq_convert(dq, B, Hq, Hkv, N, d, float(scale), workspace, workspace_bytes, stream)


def fa_strerror(status):
    return load_library().fa_strerror(status).decode()


def fa_last_device_status(stream=None):
    """Return (status, (block, site, thread))."""
    detail = (ctypes.c_int * 3)()
    s = load_library().fa_last_device_status(stream, detail)
    return s, tuple(detail)


def fa_selftest_wait_timeout(timeout_ns, stream=None):
    return load_library().fa_selftest_wait_timeout(int(timeout_ns), stream)


def fa_selftest_drain_timeout(timeout_ns, stream=None):
    return load_library().fa_selftest_drain_timeout(int(timeout_ns), stream)


def fa_version():
    return load_library().fa_version()


def fa_last_cuda_error():
    return load_library().fa_last_cuda_error().decode()


def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, causal, scale, stream):
    """fa_bwd without a workspace argument: the scratch is a fixed buffer inside
    the library (for callers that cannot allocate device memory)."""
    return load_library().fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, int(causal),
                                         float(scale), stream)


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(t, name, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(status, what):
    if status != FA_OK:
        if status in (FA_ERR_LAUNCH, FA_ERR_CUDA):
            what = f"{what} [{fa_last_cuda_error()}]"
        raise FAError(status, what)


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None):
    """O, LSE = exact attention of bf16 [B,Hq,N,d] q and [B,Hkv,N,d] k, v."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    _check(q, "q", (B, Hq, N, d), torch.bfloat16)
    _check(k, "k", (B, Hkv, N, d), torch.bfloat16)
    _check(v, "v", (B, Hkv, N, d), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    _check(out, "out", (B, Hq, N, d), torch.bfloat16)
    _check(lse, "lse", (B, Hq, N), torch.float32)
    _raise(fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                  B, Hq, Hkv, N, d, causal, scale, _stream_handle(stream)), "fa_fwd")
    return out, lse


def forward_ex(q, k, v, causal: bool = False, scale: float | None = None, window: int = 0, num_splits: int = 1,
               out=None, lse=None, workspace=None, stream=None):
    """O, LSE of bf16 q [B,Hq,Nq,d] against k, v [B,Hkv,Nk,d] (queries at the last
    Nq positions), with an optional sliding window and key splits; see fa_fwd_ex.
    ``num_splits=0`` takes fa_fwd_ex_default_splits."""
    import torch
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    _check(q, "q", (B, Hq, Nq, d), torch.bfloat16)
    _check(k, "k", (B, Hkv, Nk, d), torch.bfloat16)
    _check(v, "v", (B, Hkv, Nk, d), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits == 0:
        num_splits = fa_fwd_ex_default_splits(B, Hq, Hkv, Nq, Nk, d, causal, window)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check(out, "out", (B, Hq, Nq, d), torch.bfloat16)
    _check(lse, "lse", (B, Hq, Nq), torch.float32)
    nbytes = fa_fwd_ex_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() if workspace is not None else 0
    _raise(fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nk,
                     d, causal, window, num_splits, scale, wp, wn, _stream_handle(stream)), "fa_fwd_ex")
    return out, lse


def workspace_for(B, Hq, Hkv, N, d, device):
    import torch
    nbytes = fa_bwd_workspace_bytes(B, Hq, Hkv, N, d)
    if nbytes == 0:
        raise FAError(FA_ERR_BAD_SHAPE, "fa_bwd_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, workspace=None,
             dq=None, dk=None, dv=None, stream=None, window: int = 0, deterministic: bool = False):
    """dQ, dK, dV of sum(dO * O), recomputing P from the forward's LSE."""
    import torch
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    for t, name, hh in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq)):
        _check(t, name, (B, hh, N, d), torch.bfloat16)
    _check(lse, "lse", (B, Hq, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = workspace_for(B, Hq, Hkv, N, d, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _raise(fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, causal, window, deterministic, scale,
                     workspace.data_ptr(), workspace.numel(), _stream_handle(stream)), "fa_bwd_ex")
    return dq, dk, dv


def check_device_status(stream=None):
    """Raise FAError if a kernel of this library recorded a device-side error."""
    s, detail = fa_last_device_status(_stream_handle(stream))
    if s != FA_OK:
        raise FAError(s, f"device status (block, site, thread) = {detail}")
