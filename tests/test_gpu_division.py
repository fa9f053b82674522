"""The kernels divide a sum by a runtime rank count P that is not a power of
two with Markstein's correction (gar_device.cuh, div_small) instead of the
IEEE division, and, where the mean is only stored as bf16, with a product by
the reciprocal that falls back on the correction near a bf16 rounding
boundary (div_small_bf16).  This checks, on the GPU, for every one of the
2**32 fp32 inputs and every such P up to 16, that the first returns the IEEE
division's bits (__fdiv_rn) and that the second rounds to the same bf16 --
the bit-exact Mean results rest on both."""
import ctypes
import subprocess
from pathlib import Path

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gradient_all_reduce_gb300.build import ARCH, CSRC, INCLUDE, nvcc
    lib = tmp_path_factory.mktemp("div") / "libdivcheck.so"
    r = subprocess.run([nvcc(), *ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                        f"-I{CSRC}", f"-I{INCLUDE}", str(ROOT / "tests" / "div_exhaustive.cu"),
                        "-o", str(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    dll = ctypes.CDLL(str(lib))
    dll.div_check.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong),
                              ctypes.POINTER(ctypes.c_uint)]
    dll.div_check.restype = ctypes.c_int
    return dll


@pytest.mark.parametrize("d", [3, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15])
def test_div_small_equals_ieee_division_for_every_float(checker, d):
    bad, first = ctypes.c_ulonglong(), ctypes.c_uint()
    assert checker.div_check(d, 0, ctypes.byref(bad), ctypes.byref(first)) == 0
    assert bad.value == 0, f"d={d}: {bad.value} mismatches, first x bits 0x{first.value:08x}"


@pytest.mark.parametrize("d", [3, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15])
def test_div_small_bf16_rounds_like_ieee_division_for_every_float(checker, d):
    bad, first = ctypes.c_ulonglong(), ctypes.c_uint()
    assert checker.div_check(d, 1, ctypes.byref(bad), ctypes.byref(first)) == 0
    assert bad.value == 0, f"d={d}: {bad.value} mismatches, first x bits 0x{first.value:08x}"
