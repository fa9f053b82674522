"""Loader of the device-side input generator (``synth.cu``), for tests and
the benchmark: fills torch CUDA tensors with the same bits as the host
generators of this package."""
from __future__ import annotations

import ctypes
import hashlib
import os
import shutil
import subprocess
from pathlib import Path

import workloads

HERE = Path(__file__).resolve().parent
SRC = HERE / "synth.cu"
LIB = HERE / "libgar_synth.so"
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
         "-Xcompiler", "-fPIC", "-shared"]


def build() -> Path:
    stamp = LIB.with_suffix(".stamp")
    want = hashlib.sha256(SRC.read_bytes() + " ".join(FLAGS).encode()).hexdigest()[:16]
    if LIB.exists() and stamp.exists() and stamp.read_text() == want:
        return LIB
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB.with_name(LIB.name + f".{os.getpid()}.tmp")
    subprocess.run([nvcc, *FLAGS, "-o", str(tmp), str(SRC)], check=True)
    os.replace(tmp, LIB)
    stamp.write_text(want)
    return LIB


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = ctypes.CDLL(str(build()))
        _LIB.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                    ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                    ctypes.c_void_p]
        _LIB.synth_fill.restype = ctypes.c_int
    return _LIB


def fill(t, kind: str, seed: int, std: float = 1.0, start: int = 0, stream=None) -> None:
    """Fill CUDA tensor ``t`` (float32, or int16/uint16/bfloat16 holding bf16
    bits) with draws ``start ..`` of stream ``seed``."""
    import torch
    bf16 = t.dtype in (torch.bfloat16, torch.int16, torch.uint16)
    if not bf16 and t.dtype != torch.float32:
        raise TypeError(t.dtype)
    k = {"uniform": 0, "normal": 1}[kind]
    scale = workloads.normal_scale(std) if k == 1 else 0.0
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = _lib().synth_fill(t.data_ptr(), t.numel(), seed, start, k, int(bf16), scale, s)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed ({rc})")
