"""Calls captured in a CUDA graph and replayed: the bucket step with SGD,
the no_sync micro-batches, the ZeRO-1 step and SyncBN statistics, each a
sequence of dependent calls run once on a side stream, captured in one
graph and replayed, and compared with the oracle running the sequence as
many times, bit for bit.  Every launch is a
kernel whose launch table travels in its parameters, so a replay runs the
captured calls on the captured buffers with no host work in between."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import DT, assert_bits_equal, dev, empty, replicas, to_np
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu

SIZES = [7, 4099, 70_001]


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _graph(seq):
    """seq(stream) run once on a side stream (first launches load the
    kernels), then captured in a CUDA graph, which is returned."""
    side = torch.cuda.Stream(dev())
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        seq(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        seq(torch.cuda.current_stream())
    return graph


def _grads(P, dt, seed0, offset):
    return [replicas(P, n, dt, "normal", seed0 + 100 * t, std=1e-3, offset=offset if t == 1 else 0)
            for t, n in enumerate(SIZES)]


def _grads_host(P, dt, seed0):
    return [[workloads.replica_values("normal", dt, seed0 + 100 * t + r, n, std=1e-3)
             for r in range(P)] for t, n in enumerate(SIZES)]


def _sgd_state(seed0):
    ws = [empty(n, "f32") for n in SIZES]
    for t, w in enumerate(ws):
        wgpu.fill(w, "normal", seed0 + t, std=0.02)
    vs = [torch.zeros(n, device=dev()) for n in SIZES]
    hw = [workloads.normal_f32(seed0 + t, n, std=0.02) for t, n in enumerate(SIZES)]
    hv = [np.zeros(n, np.float32) for n in SIZES]
    return ws, vs, hw, hv


@pytest.mark.parametrize("P", [2, 5, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_bucket_sgd_steps_from_a_graph(P, dt):
    """Three Mean + SGD bucket steps in one graph (write-back on, so each
    step reduces what the one before wrote), replayed twice after the
    side-stream run: nine steps."""
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        ts = _grads(P, dt, 10 + P, offset=1)
        ws, vs, hw, hv = _sgd_state(200)

        def seq(s):
            for _ in range(3):
                gar.ar_bucket_all_reduce(comm, ts, SIZES, DT[dt], gar.AR_MEAN,
                                         sgd=(0.1, 0.9, ws, vs, 1), stream=s)

        g = _graph(seq)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    host = _grads_host(P, dt, 10 + P)
    for _ in range(9):
        oracle.bucket_all_reduce(host, op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
    for t in range(len(SIZES)):
        assert_bits_equal(to_np(ws[t]), hw[t], f"w {t}")
        assert_bits_equal(to_np(vs[t]), hv[t], f"v {t}")
        for r in range(P):
            assert_bits_equal(to_np(ts[t][r]), host[t][r], f"tensor {t} rank {r}")


@pytest.mark.parametrize("P", [2, 3, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_micro_batches_from_a_graph(P, dt):
    """One no_sync step of three micro-batches in a graph (the first, one
    before the last, and the last fused with Mean and SGD), replayed twice
    after the side-stream run: three steps, the gradients the last
    micro-batch writes back being the next step's inputs."""
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        ts = _grads(P, dt, 30 + P, offset=1)
        acc = [[torch.empty(n, device=dev()) for _ in range(P)] for n in SIZES]
        ws, vs, hw, hv = _sgd_state(400)

        def seq(s):
            gar.ar_bucket_accumulate(comm, ts, SIZES, DT[dt], acc, 1 / 3, True, s)
            gar.ar_bucket_accumulate(comm, ts, SIZES, DT[dt], acc, 1 / 3, False, s)
            gar.ar_bucket_all_reduce_accumulated(comm, ts, SIZES, DT[dt], acc, 1 / 3, False,
                                                 gar.AR_MEAN, sgd=(0.1, 0.9, ws, vs, 1),
                                                 stream=s)

        g = _graph(seq)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    host = _grads_host(P, dt, 30 + P)
    hacc = [[np.zeros(n, np.float32) for _ in range(P)] for n in SIZES]
    for _ in range(3):
        oracle.bucket_accumulate(host, hacc, 1 / 3, True)
        oracle.bucket_accumulate(host, hacc, 1 / 3, False)
        oracle.bucket_all_reduce_accumulated(host, hacc, 1 / 3, False, oracle.MEAN,
                                             sgd=(0.1, 0.9, hw, hv, 1))
    for t in range(len(SIZES)):
        assert_bits_equal(to_np(ws[t]), hw[t], f"w {t}")
        assert_bits_equal(to_np(vs[t]), hv[t], f"v {t}")
        for r in range(P):
            assert_bits_equal(to_np(ts[t][r]), host[t][r], f"tensor {t} rank {r}")
            assert_bits_equal(to_np(acc[t][r]), hacc[t][r], f"acc {t} rank {r}")


@pytest.mark.parametrize("P", [3, 8])
def test_zero1_steps_from_a_graph(P):
    """Two ZeRO-1 steps in a graph, replayed twice (six steps with the
    side-stream run), bf16 gradients fixed, fp32 shards carried over."""
    n = P * 8 * 1001 + P * 8
    sh = n // P
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        g = replicas(P, n, "bf16", "normal", 50 + P, std=1e-3)
        params = [empty(n, "bf16") for _ in range(P)]
        ws = [empty(sh, "f32") for _ in range(P)]
        for r, w in enumerate(ws):
            wgpu.fill(w, "normal", 600 + r, std=0.02)
        vs = [torch.zeros(sh, device=dev()) for _ in range(P)]

        def seq(s):
            for _ in range(2):
                gar.ar_sharded_sgd_step(comm, g, params, ws, vs, n, gar.AR_BF16, 0.1, 0.9,
                                        gar.AR_MEAN, s)

        gr = _graph(seq)
        for _ in range(2):
            gr.replay()
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    hg = [workloads.replica_values("normal", "bf16", 50 + P + r, n, std=1e-3) for r in range(P)]
    hp = [np.zeros(n, np.uint16) for _ in range(P)]
    hw = [workloads.normal_f32(600 + r, sh, std=0.02) for r in range(P)]
    hv = [np.zeros(sh, np.float32) for _ in range(P)]
    for _ in range(6):
        oracle.sharded_sgd_step(hg, hp, hw, hv, 0.1, 0.9, oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(params[r]), hp[r], f"params {r}")
        assert_bits_equal(to_np(ws[r]), hw[r], f"w shard {r}")
        assert_bits_equal(to_np(vs[r]), hv[r], f"v shard {r}")


def test_syncbn_chain_from_a_graph():
    """Twenty SyncBN statistics calls in one graph, each on the outputs'
    buffers of the one before as its sums (so each depends on the last),
    against the oracle run twenty times the same way."""
    P, C = 8, 515
    rng = np.random.default_rng(7)
    counts = [int(c) for c in rng.integers(1, 3000, size=P)]
    sums = [np.float32(rng.normal(0, 1, C) * c) for c in counts]
    sq = [np.float32(np.abs(rng.normal(1, 0.5, C)) * c + s * s / c) for s, c in zip(sums, counts)]
    d_s = [torch.from_numpy(x).to(dev()) for x in sums]
    d_q = [torch.from_numpy(x).to(dev()) for x in sq]
    d_m = [torch.empty(C, device=dev()) for _ in range(P)]
    d_i = [torch.empty(C, device=dev()) for _ in range(P)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        def seq(s):
            for k in range(20):
                a, b = (d_s, d_m) if k % 2 == 0 else (d_m, d_s)
                gar.ar_syncbn_stats(comm, a, d_q, counts, b, d_i, C, 1e-5, s)

        # Run the chain once on the side stream from the original sums,
        # then restore them before capturing.
        keep = [x.clone() for x in d_s]
        g = _graph(seq)
        for x, k in zip(d_s, keep):
            x.copy_(k)
        g.replay()
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    hs = [x.copy() for x in sums]
    hm = None
    for k in range(20):
        src = hs if k % 2 == 0 else hm
        m, i = oracle.syncbn_stats(src, sq, counts, eps=1e-5)
        if k % 2 == 0:
            hm = m
        else:
            hs = m
        hi = i
    for r in range(P):
        assert_bits_equal(to_np(d_s[r]), hs[r], f"sums {r}")
        assert_bits_equal(to_np(d_m[r]), hm[r], f"means {r}")
        nan = np.isnan(hi[r])
        assert np.array_equal(nan, np.isnan(to_np(d_i[r])))
        assert_bits_equal(to_np(d_i[r])[~nan], hi[r][~nan], f"invstd {r}")
