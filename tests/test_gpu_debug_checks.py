"""The debug build's device-side index checks.

``build(debug=True)`` compiles the library with GAR_DEBUG=1: every
register-staged kernel (reduce, copy, both accumulation kernels, SyncBN
statistics) checks each segment, tile and index against the launch's own
table before it loads or stores, and a failed check sets a bit of the
comm's status word and skips the access instead of trapping.  This test
builds that library and runs the collective, bucket, accumulation, ZeRO-1,
SyncBN, reducer, guard-band and every-rank-count parity tests against it in
a child process: they must pass against the oracle as before, with every
comm's status still AR_OK when it is destroyed (tests/debug_status_plugin.py),
and the child must have loaded the debug library and not the release one."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["test_gpu_collectives.py", "test_gpu_buckets.py", "test_gpu_accumulate.py",
         "test_gpu_sharded.py", "test_gpu_syncbn.py", "test_gpu_reducer.py",
         "test_gpu_guard_bands.py", "test_gpu_every_rank_count.py"]


def test_parity_cases_pass_under_the_debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gradient_all_reduce_gb300.build import build
    build(debug=True)
    env = dict(os.environ, GAR_LIBRARY="debug",
               PYTHONPATH=os.pathsep.join([os.path.join(ROOT, "tests"), ROOT,
                                           os.environ.get("PYTHONPATH", "")]))
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-s", "-m", "gpu", "-p", "no:cacheprovider",
           "-p", "debug_status_plugin", *[os.path.join("tests", f) for f in FILES]]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "loaded ['libgar_debug.so']" in r.stdout, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
