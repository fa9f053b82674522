"""GPU parity of the ZeRO-1 sharded SGD step (ar_sharded_sgd_step: reduce-
scatter, owner's SGD on its fp32 shard, all-gather of the updated weights,
in one pass) against the CPU oracle, bit for bit, and its equivalence with
the replicated bucketed step."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import (DT, assert_bits_equal, bits_equal_device, dev, empty, gather, host_replicas,
                     replicas, sample_indices, to_np)
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _shards(P, s, off=0):
    ws = [empty(s, "f32", off) for _ in range(P)]
    for r, w in enumerate(ws):
        wgpu.fill(w, "normal", 300 + r, std=0.02)
    vs = [torch.zeros(s + off, device=dev())[off:] for _ in range(P)]
    hw = [workloads.normal_f32(300 + r, s, std=0.02) for r in range(P)]
    hv = [np.zeros(s, np.float32) for _ in range(P)]
    return ws, vs, hw, hv


@pytest.mark.parametrize("P", [2, 3, 4, 6, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shard", [1, 5, 4096, 33_331])
@pytest.mark.parametrize("in_place", [False, True])
def test_sharded_step_equals_oracle(P, dt, shard, in_place):
    n = shard * P
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    ws, vs, hw, hv = _shards(P, shard)
    try:
        for step in range(2):
            g = replicas(P, n, dt, "normal", 40 + 10 * step, std=1e-3)
            hg = host_replicas(P, n, dt, "normal", 40 + 10 * step, std=1e-3)
            params = g if in_place else [empty(n, dt) for _ in range(P)]
            hp = [np.zeros(n, hg[0].dtype) for _ in range(P)]
            gar.ar_sharded_sgd_step(comm, g, params, ws, vs, n, DT[dt], 0.1, 0.9, gar.AR_MEAN)
            torch.cuda.synchronize()
            oracle.sharded_sgd_step(hg, hp, hw, hv, 0.1, 0.9, op=oracle.MEAN)
            for r in range(P):
                assert_bits_equal(to_np(ws[r]), hw[r], f"step {step} w {r}")
                assert_bits_equal(to_np(vs[r]), hv[r], f"step {step} v {r}")
                assert_bits_equal(to_np(params[r]), hp[r], f"step {step} params {r}")
    finally:
        gar.ar_destroy(comm)


def test_sharded_step_unaligned():
    P, shard = 4, 1001
    n = P * shard
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    ws, vs, hw, hv = _shards(P, shard, off=1)
    try:
        g = replicas(P, n, "bf16", "normal", 5, std=1e-3, offset=1)
        params = [empty(n, "bf16", 1) for _ in range(P)]
        gar.ar_sharded_sgd_step(comm, g, params, ws, vs, n, gar.AR_BF16, 0.1, 0.9, gar.AR_SUM)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    hg = host_replicas(P, n, "bf16", "normal", 5, std=1e-3)
    hp = [np.zeros(n, np.uint16) for _ in range(P)]
    oracle.sharded_sgd_step(hg, hp, hw, hv, 0.1, 0.9, op=oracle.SUM)
    for r in range(P):
        assert_bits_equal(to_np(params[r]), hp[r], f"params {r}")


def test_sharded_vit_equals_replicated_step():
    """ViT-B/16's 86,567,656 bf16 gradients as one flat unit, P=8: the
    sharded step's params equal bf16(w) of the replicated bucketed step (the
    same fp32 master weights, unsharded), on the device; sampled values
    equal the oracle's."""
    P = 8
    n = workloads.VIT_B16_PARAMS
    s = n // P
    g1 = replicas(P, n, "bf16", "normal", workloads.VIT_GRAD_SEED, std=workloads.VIT_GRAD_STD)
    g2 = [x.clone() for x in g1]
    w = empty(n, "f32")
    wgpu.fill(w, "normal", workloads.VIT_MASTER_SEED, std=workloads.VIT_MASTER_STD)
    ws = [w[r * s:(r + 1) * s].clone() for r in range(P)]
    vs = [torch.zeros(s, device=dev()) for _ in range(P)]
    v = torch.zeros(n, device=dev())
    params = [empty(n, "bf16") for _ in range(P)]
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        gar.ar_sharded_sgd_step(comm, g1, params, ws, vs, n, gar.AR_BF16, 0.1, 0.9, gar.AR_MEAN)
        gar.ar_bucket_all_reduce(comm, [g2], [n], gar.AR_BF16, gar.AR_MEAN,
                                 sgd=(0.1, 0.9, [w], [v], 0))
        torch.cuda.synchronize()
        assert bits_equal_device(torch.cat(ws), w)
        assert bits_equal_device(torch.cat(vs), v)
        wb = w.to(torch.bfloat16)      # torch's cast: round to nearest even
        for r in range(P):
            assert bits_equal_device(params[r], wb), r
    finally:
        gar.ar_destroy(comm)
    idx = sample_indices(n, 50_000, 7, extra=[s - 1, s, 7 * s])
    cols = host_replicas(P, 0, "bf16", "normal", workloads.VIT_GRAD_SEED,
                         std=workloads.VIT_GRAD_STD, idx=idx)
    hw = [workloads.normal_f32(workloads.VIT_MASTER_SEED, 0, std=workloads.VIT_MASTER_STD, idx=idx)]
    hv = [np.zeros(idx.size, np.float32)]
    ref = [[c.copy() for c in cols]]
    oracle.bucket_all_reduce(ref, op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 0))
    assert_bits_equal(gather(params[3], idx), oracle.f32_to_bf16(hw[0]), "sampled params")
