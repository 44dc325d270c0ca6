"""The store kernel's quotient x / scale is computed without a per-element
IEEE division: one correctly rounded reciprocal per tile, then Markstein's
correction (P. Markstein, IBM J. Res. Dev. 34(1), 1990) on packed f32x2.
The tile's scale (Markstein's correction with the constant RN(1/448)) and
its reciprocal (one Newton-Raphson step from the hardware approximation)
take no IEEE division either; the first test compares both with CUDA's
__fdiv_rn and __frcp_rn for every tile maximum.

This test sweeps every (value, tile maximum) pair the kernel can meet, all
finite bf16 maxima M and every bf16 x with |x| <= M (about 1.07e9 values),
and requires the E4M3 codes to equal those from CUDA's correctly rounded
__fdiv_rn.  Together with the oracle parity tests (which compare against a
true IEEE division on the CPU) this pins the arithmetic exactly."""

import ctypes
import os
import subprocess

import pytest

from replication_token_warp_gb300 import build as kbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cuda", "division_sweep.cu")
OUT_DIR = os.path.join(HERE, "_build")


@pytest.fixture(scope="module")
def sweep_lib(cuda_device):
    os.makedirs(OUT_DIR, exist_ok=True)
    so = os.path.join(OUT_DIR, "libdivision_sweep.so")
    cmd = [kbuild.nvcc(), *kbuild.NVCC_FLAGS, "-I", kbuild.CSRC, "-o", so, SRC]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.kvpub_test_division_sweep.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    lib.kvpub_test_division_sweep.restype = ctypes.c_int
    lib.kvpub_test_scale_sweep.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    lib.kvpub_test_scale_sweep.restype = ctypes.c_int
    return lib


def test_tile_scale_and_reciprocal_equal_ieee_for_every_maximum(sweep_lib):
    out = (ctypes.c_ulonglong * 10)()
    assert sweep_lib.kvpub_test_scale_sweep(out) == 0
    scale_bad = [hex(out[2 + k]) for k in range(min(out[0], 4))]
    rcp_bad = [hex(out[6 + k]) for k in range(min(out[1], 4))]
    assert out[0] == 0, f"{out[0]} scales differ from __fdiv_rn; maxima {scale_bad}"
    assert out[1] == 0, f"{out[1]} reciprocals differ from __frcp_rn; maxima {rcp_bad}"


def test_fast_quotient_codes_equal_ieee_division_everywhere(sweep_lib):
    out = (ctypes.c_ulonglong * 17)()
    assert sweep_lib.kvpub_test_division_sweep(out) == 0
    mismatches, checked = out[0], out[1]
    # 2 signs x sum over M of (M + 1) values, M over 0 .. 0x7F7F, rounded to
    # whole words of two values
    assert checked > 1.0e9
    examples = [(hex(out[3 + 2 * k]), hex(out[4 + 2 * k])) for k in range(min(out[2], 7))]
    assert mismatches == 0, f"{mismatches} words differ; first (M, x): {examples}"
