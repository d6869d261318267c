"""The C ABI from C: tests/c/fa_c_client.c links libfa_gb300.so through
include/fa.h alone.  It is compiled here (no GPU needed) and run on the GPU."""
import os
import shutil
import subprocess

import pytest

import exact_io_aware_flashattention_gb300 as fa
from exact_io_aware_flashattention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "fa_c_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_client(tmp_path):
    _build.build()
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(fa.LIB_PATH)
    exe = os.path.join(str(tmp_path), "fa_c_client")
    cmd = [cc, "-O1", "-std=c11", SRC, "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-l:libfa_gb300.so", f"-Wl,-rpath,{libdir}", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(compile_client(tmp_path))


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    exe = compile_client(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
    assert "fa_c_client ok" in r.stdout
