"""Build libfa_gb300.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

The translation units are compiled in parallel, then linked into
``exact_io_aware_flashattention_gb300/_lib/libfa_gb300.so`` with the CUDA
runtime linked statically.  ``ptxas -v`` output (registers, shared memory,
spills) is kept next to the library as ``ptxas.txt``.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_bwd_dq.cu"]
HEADERS = ["sm103a.cuh", "fa_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, "fa.h"), os.path.abspath(__file__)]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr + r.stdout


# The forward kernel splits its launch allocation between warpgroups with
# setmaxnreg; the split is only valid for this per-thread register count.
FWD_KERNEL_REGS = 168


def check_registers(ptxas_log: str) -> None:
    """Fail the build if ptxas did not give every forward-kernel instance
    exactly FWD_KERNEL_REGS registers (or spilled in it)."""
    entry = None
    seen = 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            entry = m.group(1)
            continue
        if entry and "fa_fwd_kernel" in entry:
            m = re.search(r"Used (\d+) registers", line)
            if m:
                seen += 1
                if int(m.group(1)) != FWD_KERNEL_REGS:
                    raise RuntimeError(f"{entry}: ptxas used {m.group(1)} registers, the warpgroup register split "
                                       f"needs exactly {FWD_KERNEL_REGS}")
                entry = None
            m = re.search(r"(\d+) bytes spill stores", line)
            if m and int(m.group(1)) != 0:
                raise RuntimeError(f"{entry}: {m.group(1)} bytes of register spills")
    if seen == 0:
        raise RuntimeError("ptxas reported no forward-kernel instance")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    with open(os.path.join(OUT_DIR, "ptxas.txt"), "w") as f:
        for (o, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    check_registers(results[SOURCES.index("fa_fwd.cu")][1])
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(open(os.path.join(OUT_DIR, "ptxas.txt")).read(), file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
