"""ar_all_reduce_noalloc: the all-reduce for callers that may not allocate
device memory themselves (a host framework that owns every allocation
through its own pool, a service that forbids allocations after start-up,
a hard memory cap) and therefore cannot create a comm with ar_init.

Through the C ABI, two calls in a row of the allocation-free entry point
must give exactly the bits that the regular ar_all_reduce gives on the same
inputs (the tests' tolerance for the all-reduce is bit-exact).  The file is
named to run last, and the test stands alone: it works in a fresh process
(the first call sets the device up) and after every other test."""
import pytest
import torch

import gradient_all_reduce_gb300 as gar
from gpucase import DT, OP, assert_bits_equal, empty, replicas, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_no_alloc_matches_all_reduce_twice(dt):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
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


def test_no_alloc_refuses_bad_arguments():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    xs = replicas(2, 64, "f32", "uniform", 1)
    for bad in [(0, xs, xs, 64, gar.AR_F32, gar.AR_SUM),           # no ranks
                (2, xs, xs, 64, gar.AR_F32, gar.AR_OP_DEFAULT),    # no comm, no default op
                (2, xs, [xs[1], xs[0]], 64, gar.AR_F32, gar.AR_SUM)]:  # recv aliases another send
        with pytest.raises(gar.GarError) as e:
            gar.ar_all_reduce_noalloc(*bad)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
