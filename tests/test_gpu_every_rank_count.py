"""Every rank count has a compile-time kernel of its own (P = 1 .. 16, for
the flat all-reduce in both tile sizes, the bucket step fused with SGD, the
ZeRO-1 step and the last no_sync micro-batch), so every P is run here
through each of them and compared with the CPU oracle bit for bit, with
ragged tails and one segment that is not 16-byte aligned."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import DT, assert_bits_equal, dev, empty, host_replicas, replicas, to_np
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu

ALL_P = list(range(1, 17))


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _comm(P, small_bytes=None):
    """A comm; small_bytes = 0 turns off the one-vector tiles of small flat
    all-reduces (read at init), so a small message runs the default tile."""
    import os
    old = os.environ.get("GAR_SMALL_ALL_REDUCE_BYTES")
    if small_bytes is not None:
        os.environ["GAR_SMALL_ALL_REDUCE_BYTES"] = str(small_bytes)
    try:
        return gar.ar_init(P, 0, gar.AR_MEAN)
    finally:
        if old is None:
            os.environ.pop("GAR_SMALL_ALL_REDUCE_BYTES", None)
        else:
            os.environ["GAR_SMALL_ALL_REDUCE_BYTES"] = old


@pytest.mark.parametrize("P", ALL_P)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("tile", ["one vector", "default"])
def test_flat_all_reduce_both_tiles(P, dt, tile):
    """Mean out of place and Sum in place, with the small-message tile (one
    vector per thread) and with the kernel's default unroll."""
    comm = _comm(P, None if tile == "one vector" else 0)
    try:
        n = 70_001
        for op, place, seed in (("mean", "out", 300 + P), ("sum", "in", 400 + P)):
            xs = replicas(P, n, dt, "uniform", seed)
            ys = xs if place == "in" else [empty(n, dt) for _ in range(P)]
            gar.ar_all_reduce(comm, xs, ys, n, DT[dt], gar.AR_MEAN if op == "mean" else gar.AR_SUM)
            torch.cuda.synchronize()
            assert gar.ar_get_async_error(comm) == gar.AR_OK
            want = oracle.all_reduce(host_replicas(P, n, dt, "uniform", seed),
                                     op=oracle.MEAN if op == "mean" else oracle.SUM)
            for r in range(P):
                assert_bits_equal(to_np(ys[r]), want[r], f"{op} {place} rank {r}")
    finally:
        gar.ar_destroy(comm)


SIZES = [5, 1000, 65_536 + 13]


def _grads(P, dt, seed0, offset=0):
    return [replicas(P, n, dt, "normal", seed0 + 100 * t, std=1e-3, offset=offset if t == 1 else 0)
            for t, n in enumerate(SIZES)]


def _grads_host(P, dt, seed0):
    return [[workloads.replica_values("normal", dt, seed0 + 100 * t + r, n, std=1e-3)
             for r in range(P)] for t, n in enumerate(SIZES)]


@pytest.mark.parametrize("P", ALL_P)
def test_bucket_mean_sgd(P):
    """bf16 bucket, Mean fused with SGD and write-back; tensor 1 unaligned."""
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        ts = _grads(P, "bf16", 40 + P, offset=1)
        ws = [empty(n, "f32") for n in SIZES]
        for t, w in enumerate(ws):
            wgpu.fill(w, "normal", 500 + t, std=0.02)
        vs = [torch.zeros(n, device=dev()) for n in SIZES]
        for _ in range(2):
            gar.ar_bucket_all_reduce(comm, ts, SIZES, gar.AR_BF16, gar.AR_MEAN,
                                     sgd=(0.1, 0.9, ws, vs, 1))
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    host = _grads_host(P, "bf16", 40 + P)
    hw = [workloads.normal_f32(500 + t, n, std=0.02) for t, n in enumerate(SIZES)]
    hv = [np.zeros(n, np.float32) for n in SIZES]
    for _ in range(2):
        oracle.bucket_all_reduce(host, op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
    for t in range(len(SIZES)):
        assert_bits_equal(to_np(ws[t]), hw[t], f"w {t}")
        assert_bits_equal(to_np(vs[t]), hv[t], f"v {t}")
        for r in range(P):
            assert_bits_equal(to_np(ts[t][r]), host[t][r], f"tensor {t} rank {r}")


@pytest.mark.parametrize("P", ALL_P)
def test_last_micro_batch_with_sgd(P):
    """The last no_sync micro-batch (accumulators from an earlier one) fused
    with Mean and SGD, fp32 gradients."""
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        ts = _grads(P, "f32", 60 + P)
        acc = [[torch.empty(n, device=dev()) for _ in range(P)] for n in SIZES]
        for t, n in enumerate(SIZES):
            for r in range(P):
                wgpu.fill(acc[t][r], "normal", 700 + 100 * t + r, std=1e-3)
        ws = [empty(n, "f32") for n in SIZES]
        for t, w in enumerate(ws):
            wgpu.fill(w, "normal", 600 + t, std=0.02)
        vs = [torch.zeros(n, device=dev()) for n in SIZES]
        gar.ar_bucket_all_reduce_accumulated(comm, ts, SIZES, gar.AR_F32, acc, 0.5, False,
                                             gar.AR_MEAN, sgd=(0.1, 0.9, ws, vs, 1))
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    host = _grads_host(P, "f32", 60 + P)
    hacc = [[workloads.normal_f32(700 + 100 * t + r, n, std=1e-3) for r in range(P)]
            for t, n in enumerate(SIZES)]
    hw = [workloads.normal_f32(600 + t, n, std=0.02) for t, n in enumerate(SIZES)]
    hv = [np.zeros(n, np.float32) for n in SIZES]
    oracle.bucket_all_reduce_accumulated(host, hacc, 0.5, False, oracle.MEAN,
                                         sgd=(0.1, 0.9, hw, hv, 1))
    for t in range(len(SIZES)):
        assert_bits_equal(to_np(ws[t]), hw[t], f"w {t}")
        for r in range(P):
            assert_bits_equal(to_np(ts[t][r]), host[t][r], f"tensor {t} rank {r}")


@pytest.mark.parametrize("P", ALL_P)
def test_zero1_step(P):
    """ZeRO-1 sharded step (reduce-scatter, the owner's SGD, all-gather of
    the weights), bf16, a flat unit of whole vectors per shard."""
    n = P * 8 * 1001
    sh = n // P
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        g = replicas(P, n, "bf16", "normal", 80 + P, std=1e-3)
        params = [empty(n, "bf16") for _ in range(P)]
        ws = [empty(sh, "f32") for _ in range(P)]
        for r, w in enumerate(ws):
            wgpu.fill(w, "normal", 900 + r, std=0.02)
        vs = [torch.zeros(sh, device=dev()) for _ in range(P)]
        gar.ar_sharded_sgd_step(comm, g, params, ws, vs, n, gar.AR_BF16, 0.1, 0.9, gar.AR_MEAN)
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    hg = host_replicas(P, n, "bf16", "normal", 80 + P, std=1e-3)
    hp = [np.zeros(n, np.uint16) for _ in range(P)]
    hw = [workloads.normal_f32(900 + r, sh, std=0.02) for r in range(P)]
    hv = [np.zeros(sh, np.float32) for _ in range(P)]
    oracle.sharded_sgd_step(hg, hp, hw, hv, 0.1, 0.9, oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(params[r]), hp[r], f"params {r}")
        assert_bits_equal(to_np(ws[r]), hw[r], f"w shard {r}")
