"""The C ABI from a plain C program (tests/c/abi_check.c), linked directly
against libkvpub.so: host-side validation on the CPU, and a cudaMalloc'd
three-replica store compared byte for byte with the C oracle on the GPU."""

import os
import subprocess

import pytest

import oracle
from replication_token_warp_gb300 import build as kbuild

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "abi_check.c")
OUT = os.path.join(HERE, "_build")
CUDA_HOME = os.path.dirname(os.path.dirname(kbuild.nvcc()))


def _compile(gpu: bool) -> str:
    os.makedirs(OUT, exist_ok=True)
    lib_dir = os.path.dirname(kbuild.build())
    exe = os.path.join(OUT, "abi_check_gpu" if gpu else "abi_check_cpu")
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Wextra", "-I", kbuild.INCLUDE, "-o", exe, SRC,
           "-L", lib_dir, "-lkvpub", f"-Wl,-rpath,{lib_dir}"]
    if gpu:
        oracle_dir = os.path.dirname(oracle.build())
        cmd += ["-DKVPUB_ABI_CHECK_GPU", "-I", os.path.join(CUDA_HOME, "include"),
                "-L", oracle_dir, "-lkvpub_oracle", f"-Wl,-rpath,{oracle_dir}",
                "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
                f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_program_gets_the_documented_statuses():
    exe = _compile(gpu=False)
    res = subprocess.run([exe, "cpu"], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "cpu checks ok" in res.stdout


@pytest.mark.gpu
def test_c_program_store_matches_the_oracle(cuda_device):
    exe = _compile(gpu=True)
    res = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "byte-exact" in res.stdout
