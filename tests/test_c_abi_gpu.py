"""The ABI from plain C: compile tests/c/abi_roundtrip.c with gcc against include/zpp.h,
link libzpp.so and the CUDA runtime, and run it (hand-derived expectations inside)."""
import os
import shutil
import subprocess

import pytest

from quantized_zero_communication_gb300 import build as zbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _compile(tmp_path):
    cuda = _cuda_home()
    exe = str(tmp_path / "abi_roundtrip")
    libdir = os.path.dirname(zbuild.build())
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", os.path.join(ROOT, "tests", "c", "abi_roundtrip.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", libdir, "-lzpp", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    if not os.path.exists(os.path.join(_cuda_home(), "include", "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    _compile(tmp_path)


@pytest.mark.gpu
def test_c_program_round_trip_on_gpu(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "round trip OK" in r.stdout
