"""Build libgar.so (the C-ABI library) in-tree with nvcc for sm_103a.

Translation units compile in parallel; the link makes one shared library
with the CUDA runtime linked statically.  A stamp of the sources and flags
skips the build when nothing changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libgar.so"
LIB_DEBUG = PKG / "libgar_debug.so"

UNITS = ["gar_api.cu", "gar_noalloc.cu", "gar_reducer.cu", "gar_copy.cu", "gar_reduce_f32.cu",
         "gar_reduce_bf16.cu", "gar_sgd_f32.cu", "gar_sgd_bf16.cu", "gar_acc_f32.cu", "gar_acc_bf16.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# The kernel images are stored compressed (many specialisations, each
# loaded on first use).
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-O2", "-Xfatbin", "-compress-all", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise FileNotFoundError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stamp(extra: list[str]) -> str:
    h = hashlib.sha256()
    for p in sorted(CSRC.iterdir()):
        if p.suffix in (".cu", ".cuh", ".h", ".inc"):
            h.update(p.name.encode() + p.read_bytes())
    h.update((INCLUDE / "gar.h").read_bytes())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    return h.hexdigest()[:16]


def build(verbose: bool = False, extra_flags: list[str] | None = None, force: bool = False,
          debug: bool = False) -> Path:
    """Compile every translation unit and link ``libgar.so``; returns its path.
    ``debug``: build ``libgar_debug.so`` instead, with the kernels' device-side
    index checks compiled in (GAR_DEBUG=1)."""
    extra = list(extra_flags or [])
    lib = LIB_DEBUG if debug else LIB
    if debug:
        extra.append("-DGAR_DEBUG=1")
    stamp_file = lib.with_suffix(".stamp")
    want = _stamp(extra)
    if not force and lib.exists() and stamp_file.exists() and stamp_file.read_text() == want:
        return lib
    cc = nvcc()
    with tempfile.TemporaryDirectory(prefix="gar_build_") as tmp:
        objs = [Path(tmp) / (Path(u).stem + ".o") for u in UNITS]

        def compile_one(unit_obj):
            unit, obj = unit_obj
            cmd = [cc, *NVCC_FLAGS, *extra, "-c", str(CSRC / unit), "-o", str(obj)]
            res = subprocess.run(cmd, capture_output=True, text=True)
            return cmd, res

        with ThreadPoolExecutor(max_workers=len(UNITS)) as pool:
            results = list(pool.map(compile_one, zip(UNITS, objs)))
        for cmd, res in results:
            if verbose or res.returncode != 0:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
        tmp_lib = Path(tmp) / "libgar.so"
        cmd = [cc, *ARCH, "-shared", "-o", str(tmp_lib), *map(str, objs)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("link failed: " + " ".join(cmd))
        shutil.copyfile(tmp_lib, str(lib) + ".tmp")
        os.replace(str(lib) + ".tmp", lib)
    stamp_file.write_text(want)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else None,
                force="-f" in sys.argv))
