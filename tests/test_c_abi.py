"""The C ABI from plain C99, outside Python: tests/abi_c/tpce_c_smoke.c
includes include/tpce.h, links libtpce and the CUDA runtime, and checks the
entry points against closed forms (see the file's header). On the CPU it is
compiled and linked with -Wall -Wextra -Werror (the header is valid C99); on
a GPU the program runs."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "abi_c", "tpce_c_smoke.c")


def _cuda_home():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else "/usr/local/cuda"


def _build(out):
    from vocab_ce_gb300 import build
    lib = build.build()
    cuda = _cuda_home()
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(cuda, "include"), SRC, "-L", libdir, "-ltpce", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-lm", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_c_smoke_builds_as_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    assert os.path.exists(_build(str(tmp_path / "tpce_c_smoke")))


@pytest.mark.gpu
def test_c_smoke_runs(tmp_path):
    from _parity import gpu_or_skip
    gpu_or_skip()
    exe = _build(str(tmp_path / "tpce_c_smoke"))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "tpce C ABI smoke: ok" in r.stdout
