"""The SyncBN statistics kernel divides the pooled sums by the pooled count
with Markstein's correction applied twice and the host's RN(1/n)
(gar_device.cuh, div_count) instead of the IEEE division.  This checks it on
the GPU against __ddiv_rn, bit for bit, on 2**28 random quotients and 2**28
quotients next to a rounding midpoint (the hard cases), for counts of 1 to
53 significant bits."""
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
    lib = tmp_path_factory.mktemp("arith") / "libsyncbnarith.so"
    r = subprocess.run([nvcc(), *ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                        f"-I{CSRC}", f"-I{INCLUDE}", str(ROOT / "tests" / "syncbn_arith_check.cu"),
                        "-o", str(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    dll = ctypes.CDLL(str(lib))
    u64, pu64 = ctypes.c_ulonglong, ctypes.POINTER(ctypes.c_ulonglong)
    dll.div_count_check.argtypes = [u64, u64, ctypes.c_int, pu64, pu64]
    dll.div_count_check.restype = ctypes.c_int
    return dll


@pytest.mark.parametrize("mode", [0, 1], ids=["random", "near-midpoint"])
def test_div_count_equals_ieee_division(checker, mode):
    bad, first = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    assert checker.div_count_check(0x5EED + mode, 1 << 28, mode, ctypes.byref(bad),
                                   ctypes.byref(first)) == 0
    assert bad.value == 0, f"{bad.value} mismatches, first case {first.value}"
