"""Failure detection on the GPU without a fault: a bounded device-side wait
on an mbarrier that nothing arrives at gives up, records AR_ERR_TIMEOUT in
the comm's status word, and the context stays usable."""
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
from gpucase import PATHS, assert_bits_equal, host_replicas, init, replicas, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bounded_wait_gives_up_and_reports():
    comm = gar.ar_init(2, 0, gar.AR_SUM)
    try:
        assert gar.ar_get_async_error(comm) == gar.AR_OK
        gar.ar_selftest_wait_timeout(comm, 100)
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_ERR_TIMEOUT
        assert gar.ar_get_async_error(comm) == gar.AR_ERR_TIMEOUT   # sticky
    finally:
        gar.ar_destroy(comm)
    with pytest.raises(gar.GarError):
        c = gar.ar_init(2, 0, gar.AR_SUM)
        try:
            gar.ar_selftest_wait_timeout(c, 0)
        finally:
            gar.ar_destroy(c)


@pytest.mark.parametrize("path", PATHS)
def test_context_usable_after_timeout(path):
    """After a wait gave up, a new comm's all-reduce is still bit-exact."""
    c = gar.ar_init(2, 0, gar.AR_SUM)
    gar.ar_selftest_wait_timeout(c, 50)
    torch.cuda.synchronize()
    gar.ar_destroy(c)
    P, n = 4, 100_003
    comm = init(P, gar.AR_MEAN, path)
    try:
        xs = replicas(P, n, "f32", "uniform", 9)
        gar.ar_all_reduce(comm, xs, xs, n, gar.AR_F32, gar.AR_MEAN)
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "uniform", 9), op=oracle.MEAN)
    assert_bits_equal(to_np(xs[0]), want[0], "after timeout")
