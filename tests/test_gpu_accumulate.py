"""GPU parity of DDP's no_sync gradient accumulation through the C ABI
(ar_bucket_accumulate on the micro-batches before the last,
ar_bucket_all_reduce_accumulated on the last) against the CPU oracle, bit
for bit; and the DDP-equivalence MLP with micro-batches against the fp64
full-batch gradient."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import DT, assert_bits_equal, bits_equal_device, dev, empty, replicas, to_np
from golden import table
from oracle import mlp
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu

SIZES = [1, 7, 768, 1000, 2304 * 768, 3, 65_536 + 13]


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _micro(P, sizes, dt, m, off=0):
    """Micro-batch m's gradients: tensor t, rank r from seed 1000*m + 100*t + r."""
    return [replicas(P, n, dt, "normal", 1000 * m + 100 * t, std=1e-3, offset=off)
            for t, n in enumerate(sizes)]


def _micro_host(P, sizes, dt, m):
    return [[workloads.replica_values("normal", dt, 1000 * m + 100 * t + r, n, std=1e-3)
             for r in range(P)] for t, n in enumerate(sizes)]


@pytest.mark.parametrize("P", [2, 3, 4, 6, 8, 11, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("sgd_wb", [None, 0, 1])
@pytest.mark.parametrize("aligned", [True, False])
def test_accumulate_then_reduce_equals_oracle(P, dt, sgd_wb, aligned):
    M, scale = 3, 1.0 / 3.0
    off = 0 if aligned else 1
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    acc = [[torch.full((n + off,), 7.0, device=dev())[off:] for _ in range(P)] for n in SIZES]
    hacc = [[np.full(n, 7.0, np.float32) for _ in range(P)] for n in SIZES]
    sgd = hsgd = None
    if sgd_wb is not None:
        ws = [empty(n, "f32", off) for n in SIZES]
        for t, w in enumerate(ws):
            wgpu.fill(w, "normal", 200 + t, std=0.02)
        vs = [torch.zeros(n + off, device=dev())[off:] for n in SIZES]
        sgd = (0.1, 0.9, ws, vs, sgd_wb)
        hsgd = (0.1, 0.9, [workloads.normal_f32(200 + t, n, std=0.02) for t, n in enumerate(SIZES)],
                [np.zeros(n, np.float32) for n in SIZES], sgd_wb)
    try:
        for m in range(M):
            g = _micro(P, SIZES, dt, m, off)
            hg = _micro_host(P, SIZES, dt, m)
            if m < M - 1:
                gar.ar_bucket_accumulate(comm, g, SIZES, DT[dt], acc, scale, m == 0)
                oracle.bucket_accumulate(hg, hacc, scale, m == 0)
                torch.cuda.synchronize()
                for t in range(len(SIZES)):
                    for r in (0, P - 1):
                        assert_bits_equal(to_np(acc[t][r]), hacc[t][r], f"acc m{m} t{t} r{r}")
            else:
                gar.ar_bucket_all_reduce_accumulated(comm, g, SIZES, DT[dt], acc, scale, False,
                                                     gar.AR_MEAN, sgd=sgd)
                oracle.bucket_all_reduce_accumulated(hg, hacc, scale, False, op=oracle.MEAN,
                                                     sgd=hsgd)
                torch.cuda.synchronize()
                assert gar.ar_get_async_error(comm) == gar.AR_OK
                for t in range(len(SIZES)):
                    for r in (0, P - 1):
                        assert_bits_equal(to_np(g[t][r]), hg[t][r], f"grad t{t} r{r}")
                    if sgd is not None:
                        assert_bits_equal(to_np(sgd[2][t]), hsgd[2][t], f"w t{t}")
                        assert_bits_equal(to_np(sgd[3][t]), hsgd[3][t], f"v t{t}")
    finally:
        gar.ar_destroy(comm)


def test_single_micro_batch_is_the_bucket_all_reduce():
    """first = 1, scale = 1 gives exactly ar_bucket_all_reduce's bits; the
    accumulators are not written."""
    P = 4
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        a = _micro(P, SIZES, "bf16", 5)
        b = _micro(P, SIZES, "bf16", 5)
        acc = [[torch.full((n,), 7.0, device=dev()) for _ in range(P)] for n in SIZES]
        gar.ar_bucket_all_reduce(comm, a, SIZES, gar.AR_BF16, gar.AR_MEAN)
        gar.ar_bucket_all_reduce_accumulated(comm, b, SIZES, gar.AR_BF16, acc, 1.0, True,
                                             gar.AR_MEAN)
        torch.cuda.synchronize()
        for t in range(len(SIZES)):
            for r in range(P):
                assert bits_equal_device(a[t][r], b[t][r]), (t, r)
                assert bool(torch.all(acc[t][r] == 7.0))
    finally:
        gar.ar_destroy(comm)


def test_many_tensors_split_launches():
    """300 tensors x P=8 (more segments than one parameter block holds)."""
    P, M = 8, 2
    rng = np.random.default_rng(3)
    sizes = [int(s) for s in rng.integers(1, 500, size=300)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        acc = [[torch.zeros(n, device=dev()) for _ in range(P)] for n in sizes]
        hacc = [[np.zeros(n, np.float32) for _ in range(P)] for n in sizes]
        g0, h0 = _micro(P, sizes, "f32", 0), _micro_host(P, sizes, "f32", 0)
        gar.ar_bucket_accumulate(comm, g0, sizes, gar.AR_F32, acc, 0.5, True)
        oracle.bucket_accumulate(h0, hacc, 0.5, True)
        g1, h1 = _micro(P, sizes, "f32", 1), _micro_host(P, sizes, "f32", 1)
        gar.ar_bucket_all_reduce_accumulated(comm, g1, sizes, gar.AR_F32, acc, 0.5, False,
                                             gar.AR_SUM)
        oracle.bucket_all_reduce_accumulated(h1, hacc, 0.5, False, op=oracle.SUM)
        torch.cuda.synchronize()
        for t in range(0, len(sizes), 7):
            assert_bits_equal(to_np(g1[t][P - 1]), h1[t][P - 1], f"t{t}")
    finally:
        gar.ar_destroy(comm)


def test_accumulation_ddp_equivalence_mlp():
    """The DDP-equivalence MLP, each rank's 128 rows in 2 micro-batches of 64
    (fp64 gradients rounded to fp32, host): accumulate with scale 1/2, then
    all-reduce (Mean) on the last micro-batch on the GPU; bit-exact with the
    oracle and within 1e-5 of the fp64 full-batch gradient."""
    ws, x, t = workloads.mlp_problem()
    P, M = workloads.MLP_SHARDS, 2
    full = mlp.forward_backward(ws, x, t)[1]
    rows = x.shape[0] // (P * M)
    host = []
    for m in range(M):
        per = [mlp.forward_backward(ws, x[(r * M + m) * rows:(r * M + m + 1) * rows],
                                    t[(r * M + m) * rows:(r * M + m + 1) * rows])[1]
               for r in range(P)]
        host.append([[np.ascontiguousarray(per[r][k], np.float32).ravel() for r in range(P)]
                     for k in range(len(ws))])
    sizes = [h[0].size for h in host[0]]
    dev_g = [[[torch.from_numpy(a).to(dev()) for a in reps] for reps in hm] for hm in host]
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        acc = [[torch.empty(n, device=dev()) for _ in range(P)] for n in sizes]
        gar.ar_bucket_accumulate(comm, dev_g[0], sizes, gar.AR_F32, acc, 0.5, True)
        gar.ar_bucket_all_reduce_accumulated(comm, dev_g[1], sizes, gar.AR_F32, acc, 0.5, False,
                                             gar.AR_MEAN)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    hacc = [[np.zeros(n, np.float32) for _ in range(P)] for n in sizes]
    oracle.bucket_accumulate(host[0], hacc, 0.5, True)
    oracle.bucket_all_reduce_accumulated(host[1], hacc, 0.5, False, op=oracle.MEAN)
    for k in range(len(ws)):
        assert_bits_equal(to_np(dev_g[1][k][0]), host[1][k][0], f"layer {k}")
    got = [to_np(dev_g[1][k][0]).reshape(full[k].shape) for k in range(len(ws))]
    err = mlp.linf_rel(got, full)
    assert err <= float(table("ddp_equivalence.txt")["accept"]), err
