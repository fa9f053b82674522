"""The multi-rank logic of bench.py on CPU with the gloo backend (world
size 2): every rank sees the maximum of the per-rank times, the barrier
returns on both, and only rank 0 runs the CPU reference arm."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    got = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    out.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.parametrize("case", ["ar", "rs", "ag", "bc", "zero1", "sgd", "accfirst", "acc",
                                  "acclast", "syncbn"])
def test_case_cpu_baseline_runs_every_case(case):
    """The oracle beside each --case line runs on the host for every case,
    at a P that is not a power of two, and reports a positive rate."""
    sys.path.insert(0, ROOT)
    import bench
    got = bench.case_cpu_baseline(case, 6, "bf16", "mean", min_seconds=0.0)
    assert got["kind"] == "oracle" and got["cores"] == 1 and got["unit"] == "GB/s"
    assert got["value"] > 0 and "P=6" in got["sample"]


def test_reference_arm_never_loads_the_cuda_library():
    """The oracle arm runs without the product: after a full --impl
    reference run the CUDA library's package was never imported, and the
    line carries the same config as the GPU arm's."""
    code = ("import runpy, sys, json, io, contextlib\n"
            "sys.argv = ['bench.py', '--impl', 'reference', '--steps', '2', '--warmup', '1',"
            " '--ref-budget', '0.3']\n"
            "buf = io.StringIO()\n"
            "with contextlib.redirect_stdout(buf):\n"
            "    runpy.run_path('bench.py', run_name='__main__')\n"
            "line = json.loads(buf.getvalue().strip().splitlines()[-1])\n"
            "print(json.dumps({'loaded': 'gradient_all_reduce_gb300' in sys.modules,"
            " 'line': line}))\n")
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["loaded"] is False
    line = out["line"]
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["cores"] >= 1 and line["cpu_baseline"]["kind"] == "oracle"
    sys.path.insert(0, ROOT)
    import bench
    assert line["config"] == bench.vit_config(1)


def test_threaded_oracle_step_is_bit_identical_to_one_call():
    """The all-cores CPU baseline calls the unchanged oracle from several
    threads on disjoint element ranges; the step is elementwise, so every
    output bit (gradients written back, master weights, momentum) equals
    one call over all elements, over three consecutive steps."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    n = 300_007
    one = bench.oracle_inputs(n, offset=1 << 20, threads=3)
    many = ([g.copy() for g in one[0]], one[1].copy(), one[2].copy())
    with ThreadPoolExecutor(7) as pool:
        for _ in range(3):
            bench.oracle_step(one, 1)
            bench.oracle_step(many, 7, pool)
    for a, b in zip(one[0] + [one[1], one[2]], many[0] + [many[1], many[2]]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    assert not np.array_equal(one[1], bench.oracle_inputs(n, offset=1 << 20)[1])  # w moved
