"""The bulk-copy kernels on a second GPU.

Their shared-memory opt-in is an attribute of the kernel in each device's
context, and the allocation-free all-reduce sets up each device it runs on,
so the first device's set-up must not stand in for the second's.  On a
machine with more than one visible GPU this runs the bulk-copy reduce and
copy pipelines (GAR_KERNEL=tma, GAR_COPY=tma) through a comm on device 1,
and the allocation-free all-reduce with device 1 current, against the
oracle; with one GPU it is skipped."""
import os

import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import assert_bits_equal, to_np

pytestmark = pytest.mark.gpu


def _second_device():
    if not torch.cuda.is_available() or torch.cuda.device_count() < 2:
        pytest.skip("needs two CUDA devices")
    return torch.device("cuda", 1)


def _replicas(P, n, seed, device):
    host = [workloads.uniform_f32(seed + r, n) for r in range(P)]
    return host, [torch.from_numpy(h).to(device) for h in host]


def test_bulk_copy_pipelines_on_device_1():
    dev1 = _second_device()
    P, n = 4, 300_007
    keys = ("GAR_KERNEL", "GAR_COPY")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "tma"
    try:
        comm = gar.ar_init(P, 1, gar.AR_MEAN)
    finally:
        for k in keys:
            if old[k] is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = old[k]
    try:
        host, xs = _replicas(P, n, 11, dev1)
        with torch.cuda.device(1):
            gar.ar_all_reduce(comm, xs, xs, n, gar.AR_F32, gar.AR_MEAN)
            torch.cuda.synchronize(dev1)
        assert gar.ar_get_async_error(comm) == gar.AR_OK
        want = oracle.all_reduce(host, op=oracle.MEAN)
        for r in range(P):
            assert_bits_equal(to_np(xs[r]), want[r], f"all-reduce rank {r}")
        shard = n // P
        hs, ins = _replicas(P, shard, 21, dev1)
        outs = [torch.empty(shard * P, device=dev1) for _ in range(P)]
        with torch.cuda.device(1):
            gar.ar_all_gather(comm, ins, outs, shard * P, gar.AR_F32)
            torch.cuda.synchronize(dev1)
        assert gar.ar_get_async_error(comm) == gar.AR_OK
        gathered = np.concatenate(hs)
        for r in range(P):
            assert_bits_equal(to_np(outs[r]), gathered, f"all-gather rank {r}")
    finally:
        gar.ar_destroy(comm)


def test_no_alloc_on_device_1():
    dev1 = _second_device()
    P, n = 3, 200_003
    host, xs = _replicas(P, n, 31, dev1)
    ys = [torch.empty(n, device=dev1) for _ in range(P)]
    with torch.cuda.device(1):
        gar.ar_all_reduce_noalloc(P, xs, ys, n, gar.AR_F32, gar.AR_MEAN,
                                  stream=torch.cuda.current_stream(dev1))
        torch.cuda.synchronize(dev1)
    want = oracle.all_reduce(host, op=oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"rank {r}")
