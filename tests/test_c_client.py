"""The C ABI from plain C: tests/c_client.c compiles with gcc and links
against include/gar.h and libgar.so on any machine (no GPU needed), and
runs on a GPU."""
import os
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


def _build(tmp_path: Path) -> Path:
    from gradient_all_reduce_gb300.build import LIB, build, nvcc
    build()
    cuda = Path(nvcc()).resolve().parent.parent
    exe = tmp_path / "c_client"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-O1", str(ROOT / "tests" / "c_client.c"),
                        f"-I{ROOT / 'include'}", f"-I{cuda / 'include'}", str(LIB),
                        f"-Wl,-rpath,{LIB.parent}", f"-Wl,-rpath,{cuda / 'lib64'}",
                        f"-L{cuda / 'lib64'}", "-lcudart",
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert _build(tmp_path).exists()


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ))
    assert r.returncode == 0, r.stderr
    assert "c_client: ok" in r.stdout
