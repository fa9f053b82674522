"""GPU parity of the bucketed all-reduce and its fused SGD-momentum step
through the C ABI, against the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import (DT, OP, ORACLE_OP, PATHS, assert_bits_equal, dev, empty, init, replicas,
                     to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(params=PATHS)
def path(request):
    return request.param


def _bucket(P, sizes, dt, seed0, offset=0):
    """Tensor t's replica r: draws of stream seed0 + 100 t + r (device)."""
    return [replicas(P, n, dt, "normal", seed0 + 100 * t, offset=offset)
            for t, n in enumerate(sizes)]


def _host(P, sizes, dt, seed0):
    return [[workloads.replica_values("normal", dt, seed0 + 100 * t + r, n) for r in range(P)]
            for t, n in enumerate(sizes)]


SHAPES = [(1,), (7,), (768,), (1000,), (2304, 768), (3,), (65_536 + 13,)]


@pytest.mark.parametrize("P", [2, 3, 4, 6, 8, 12])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "mean"])
def test_bucket_equals_oracle(cuda, path, P, dt, op):
    sizes = [int(np.prod(s)) for s in SHAPES]
    comm = init(P, gar.AR_MEAN, path)
    try:
        ts = _bucket(P, sizes, dt, 1)
        gar.ar_bucket_all_reduce(comm, ts, sizes, DT[dt], OP[op])
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    host = _host(P, sizes, dt, 1)
    oracle.bucket_all_reduce(host, op=ORACLE_OP[op])
    for t in range(len(sizes)):
        for r in range(P):
            assert_bits_equal(to_np(ts[t][r]), host[t][r], f"tensor {t} rank {r}")


@pytest.mark.parametrize("P", [3, 6, 8, 12])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("write_back", [0, 1])
@pytest.mark.parametrize("aligned", [True, False])
def test_bucket_sgd_equals_oracle(cuda, path, P, dt, write_back, aligned):
    """Two steps of the fused Mean + SGD(momentum 0.9, lr 0.1) on fp32
    master weights ~N(0, 0.02) and zero momentum, for P = 8 and for one P
    of each bounded kernel (at most 4, 8, 16 ranks)."""
    sizes = [int(np.prod(s)) for s in SHAPES]
    off = 0 if aligned else 1
    ts = _bucket(P, sizes, dt, 2, offset=off)
    host = _host(P, sizes, dt, 2)
    ws, vs, hw, hv = [], [], [], []
    for t, n in enumerate(sizes):
        w = empty(n, "f32", off)
        from workloads import gpu as wgpu
        wgpu.fill(w, "normal", 200 + t, std=0.02)
        ws.append(w)
        vs.append(torch.zeros(n + off, dtype=torch.float32, device=dev())[off:])
        hw.append(workloads.normal_f32(200 + t, n, std=0.02))
        hv.append(np.zeros(n, np.float32))
    comm = init(P, gar.AR_MEAN, path)
    try:
        for step in range(2):
            gar.ar_bucket_all_reduce(comm, ts, sizes, DT[dt], gar.AR_MEAN,
                                     sgd=(0.1, 0.9, ws, vs, write_back))
            torch.cuda.synchronize()
            oracle.bucket_all_reduce(host, op=oracle.MEAN,
                                     sgd=(0.1, 0.9, hw, hv, write_back))
            for t in range(len(sizes)):
                assert_bits_equal(to_np(ws[t]), hw[t], f"step {step} w {t}")
                assert_bits_equal(to_np(vs[t]), hv[t], f"step {step} v {t}")
                for r in (0, P - 1):
                    assert_bits_equal(to_np(ts[t][r]), host[t][r], f"step {step} g {t}/{r}")
    finally:
        gar.ar_destroy(comm)


def test_bucket_larger_than_one_parameter_block(cuda, path):
    """600 small tensors at P=4 (more than one launch's segment table):
    results equal the per-tensor oracle."""
    P = 4
    rng = np.random.default_rng(0)
    sizes = [int(s) for s in rng.integers(1, 3000, size=600)]
    flat = sum(sizes)
    base = replicas(P, flat, "bf16", "normal", 300)
    ts, off = [], 0
    for n in sizes:
        ts.append([b[off:off + n] for b in base])
        off += n
    comm = init(P, gar.AR_MEAN, path)
    try:
        gar.ar_bucket_all_reduce(comm, ts, sizes, gar.AR_BF16)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    host = [workloads.replica_values("normal", "bf16", 300 + r, flat) for r in range(P)]
    want = oracle.all_reduce(host, op=oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(base[r]), want[r], f"rank {r}")


def test_bucket_rejects_overlap(cuda):
    P = 2
    x = replicas(P, 1000, "f32", "uniform", 1)
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        with pytest.raises(gar.GarError) as e:
            gar.ar_bucket_all_reduce(comm, [[x[0][:600], x[1][:600]], [x[0][500:], x[1][500:]]],
                                     [600, 500], gar.AR_F32)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
        w = torch.zeros(1000, device=dev())
        with pytest.raises(gar.GarError):
            gar.ar_bucket_all_reduce(comm, [x], [1000], gar.AR_F32,
                                     sgd=(0.1, 0.9, [w], [w], 1))   # master aliases momentum
    finally:
        gar.ar_destroy(comm)


def _allocation(ptr):
    """(base, size) of the device allocation that holds ptr, from the driver."""
    import ctypes
    drv = ctypes.CDLL("libcuda.so.1")
    base, size = ctypes.c_uint64(), ctypes.c_size_t()
    rc = drv.cuMemGetAddressRange_v2(ctypes.byref(base), ctypes.byref(size), ctypes.c_uint64(ptr))
    assert rc == 0, rc
    return base.value, size.value


def test_bounds_checked_inside_an_allocation_already_seen(cuda):
    """A call validates each device allocation once and then checks later
    buffers that start inside it against its end alone.  Tensor 0 makes the
    allocation known; tensor 1 starts inside it: ending exactly at the
    allocation's end it is accepted (and reduced), one element further it is
    refused.  Likewise for the SGD master / momentum arrays."""
    comm = gar.ar_init(1, 0, gar.AR_SUM)
    try:
        torch.cuda.empty_cache()        # fresh allocations: no other tensor inside them
        a = torch.zeros(4 << 20, device=dev())
        base, size = _allocation(a.data_ptr())
        k = 4096
        start = a.data_ptr() + 4 * k
        m = (base + size - start) // 4               # tensor 1 ends at the allocation's end
        assert m >= 1 and start + 4 * m == base + size
        ptrs = [[a.data_ptr()], [start]]
        gar.ar_bucket_all_reduce(comm, ptrs, [k, m], gar.AR_F32)
        torch.cuda.synchronize()
        with pytest.raises(gar.GarError) as e:
            gar.ar_bucket_all_reduce(comm, ptrs, [k, m + 1], gar.AR_F32)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
        with pytest.raises(gar.GarError) as e:                      # the same buffer alone
            gar.ar_bucket_all_reduce(comm, [[start]], [m + 1], gar.AR_F32)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
        # master and momentum as views of one allocation each, after the grads
        g = torch.zeros(2 * k, device=dev())
        w = torch.zeros(4 << 20, device=dev())
        wb, wsize = _allocation(w.data_ptr())
        v = torch.zeros(2 * k, device=dev())
        wend = wb + wsize
        w1 = wend - 4 * k                             # master of tensor 1: the last k floats
        assert w1 >= w.data_ptr() + 4 * k
        sgd_ok = (0.1, 0.9, [w.data_ptr(), w1], [v[:k], v[k:]], 0)
        gar.ar_bucket_all_reduce(comm, [[g[:k]], [g[k:]]], [k, k], gar.AR_F32, sgd=sgd_ok)
        torch.cuda.synchronize()
        sgd_bad = (0.1, 0.9, [w.data_ptr(), w1 + 4], [v[:k], v[k:]], 0)   # one float past
        with pytest.raises(gar.GarError) as e:
            gar.ar_bucket_all_reduce(comm, [[g[:k]], [g[k:]]], [k, k], gar.AR_F32, sgd=sgd_bad)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
