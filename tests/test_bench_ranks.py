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
