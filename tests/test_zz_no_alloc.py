"""ar_all_reduce_noalloc: the all-reduce for callers that may not allocate
device memory themselves (a host framework that owns every allocation
through its own pool, a service that forbids allocations after start-up,
a hard memory cap) and therefore cannot create a comm with ar_init.

Through the C ABI, two calls in a row of the allocation-free entry point
must give exactly the bits that the regular ar_all_reduce gives on the same
inputs (the tests' tolerance for the all-reduce is bit-exact), and the bits
of the CPU oracle for every rank count class (one rank, a count that is not
a power of two, the compile-time counts, the largest), both element types,
Sum and Mean, in and out of place, and buffers that are not 16-byte aligned
(the kernel's scalar path).  The file is named to run last, and the tests
stand alone: they work in a fresh process (the first call sets the device
up) and after every other test."""
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
from gpucase import (DT, OP, ORACLE_OP, assert_bits_equal, empty, host_replicas, replicas,
                     to_np)

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_no_alloc_matches_all_reduce_twice(dt):
    _need_gpu()
    P, n = 4, 200_003   # several tiles and a ragged tail
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        for call, (seed, op) in enumerate([(500, "mean"), (600, "sum")]):
            xs = replicas(P, n, dt, "normal", seed)
            want = [empty(n, dt) for _ in range(P)]
            gar.ar_all_reduce(comm, xs, want, n, DT[dt], OP[op])
            got = [empty(n, dt) for _ in range(P)]
            gar.ar_all_reduce_noalloc(P, xs, got, n, DT[dt], OP[op])
            torch.cuda.synchronize()
            for r in range(P):
                assert_bits_equal(to_np(got[r]), to_np(want[r]), f"call {call} rank {r}")
    finally:
        gar.ar_destroy(comm)


@pytest.mark.parametrize("P", [1, 3, 4, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "mean"])
@pytest.mark.parametrize("place", ["out", "in"])
def test_no_alloc_equals_oracle(P, dt, op, place):
    """Two calls in a row on different inputs, each against the oracle."""
    _need_gpu()
    n = 70_001
    for call in range(2):
        seed = 1000 * call + 17 * P
        xs = replicas(P, n, dt, "normal", seed)
        ys = xs if place == "in" else [empty(n, dt) for _ in range(P)]
        gar.ar_all_reduce_noalloc(P, xs, ys, n, DT[dt], OP[op])
        torch.cuda.synchronize()
        host = host_replicas(P, n, dt, "normal", seed)
        want = oracle.all_reduce(host, op=ORACLE_OP[op])
        for r in range(P):
            assert_bits_equal(to_np(ys[r]), want[r], f"call {call} rank {r}")
            if place == "out":
                assert_bits_equal(to_np(xs[r]), host[r], f"call {call} send {r} untouched")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_no_alloc_unaligned_equals_oracle(dt):
    """Buffers one element past a 16-byte boundary (the scalar path), P = 5
    (the division of a Mean over a count that is not a power of two)."""
    _need_gpu()
    P, n = 5, 33_331
    xs = replicas(P, n, dt, "uniform", 77, offset=1)
    ys = [empty(n, dt, offset=1) for _ in range(P)]
    gar.ar_all_reduce_noalloc(P, xs, ys, n, DT[dt], gar.AR_MEAN)
    torch.cuda.synchronize()
    want = oracle.all_reduce(host_replicas(P, n, dt, "uniform", 77), op=oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"rank {r}")


def test_no_alloc_refuses_bad_arguments():
    _need_gpu()
    xs = replicas(2, 64, "f32", "uniform", 1)
    for bad in [(0, xs, xs, 64, gar.AR_F32, gar.AR_SUM),           # no ranks
                (17, xs, xs, 64, gar.AR_F32, gar.AR_SUM),          # more ranks than supported
                (2, xs, xs, 64, gar.AR_F32, gar.AR_OP_DEFAULT),    # no comm, no default op
                (2, xs, [xs[1], xs[0]], 64, gar.AR_F32, gar.AR_SUM)]:  # recv aliases another send
        with pytest.raises(gar.GarError) as e:
            gar.ar_all_reduce_noalloc(*bad)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
