"""The five workloads at full size on the GPU, through the C ABI, against the
CPU oracle: the DDP-equivalence MLP step (one 16 MiB bucket, P=8), the
ViT-B/16 bucketed Mean + SGD step (P=8, bf16, 8 buckets of 25 MiB), the
large-bucket stress (P=4, 2**30 fp32 per replica: RS, AG, AR), and the
size/replica sweep (4 KiB .. 1 GiB per replica, P = 2/4/8, fp32/bf16,
Sum/Mean, broadcast).  Where the oracle cannot redo a whole output in
seconds, it recomputes sampled outputs one by one from the same seeded
inputs (regenerated on the host), and properties that hold at any size are
checked on the device."""
import gc

import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import (DT, OP, ORACLE_OP, PATHS, assert_bits_equal, bits_equal_device, dev, empty,
                     gather, host_replicas, init, replicas, sample_indices, to_np)
from golden import table
from oracle import mlp
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu


@pytest.fixture(params=PATHS)
def path(request):
    return request.param


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    gc.collect()
    torch.cuda.empty_cache()


def test_ddp_equivalence_mlp(path):
    """Per-shard gradients of the 4-layer 1024-wide MLP (8 shards of 128
    rows, computed in fp64 on the host and rounded to fp32) are the P=8
    replicas; the GPU Mean over one 16 MiB bucket equals the oracle's bits
    and the fp64 full-batch gradient within 1e-5 (L-inf/L-inf)."""
    ws, x, t = workloads.mlp_problem()
    full = mlp.forward_backward(ws, x, t)[1]
    shards = mlp.shard_gradients(ws, x, t, workloads.MLP_SHARDS)
    host = [[np.ascontiguousarray(s[k], dtype=np.float32).ravel() for s in shards]
            for k in range(len(ws))]
    dev_t = [[torch.from_numpy(h).to(dev()) for h in reps] for reps in host]
    sizes = [h[0].size for h in host]
    plan = gar.ar_bucket_plan([4 * n for n in sizes], 25 << 20)
    assert plan == [0, 0, 0, 0]
    P = workloads.MLP_SHARDS
    comm = init(P, gar.AR_MEAN, path)
    try:
        gar.ar_bucket_all_reduce(comm, dev_t, sizes, gar.AR_F32, gar.AR_MEAN)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    oracle.bucket_all_reduce(host, op=oracle.MEAN)
    for k in range(len(ws)):
        for r in range(P):
            assert_bits_equal(to_np(dev_t[k][r]), host[k][r], f"layer {k} rank {r}")
    got = [to_np(dev_t[k][0]).reshape(full[k].shape) for k in range(len(ws))]
    err = mlp.linf_rel(got, full)
    assert err <= float(table("ddp_equivalence.txt")["accept"]), err


def _vit_buckets(cap):
    numels = workloads.vit_b16_numels()
    plan = gar.ar_bucket_plan([2 * n for n in numels], cap)
    offs = np.concatenate([[0], np.cumsum(numels)])
    buckets = [[] for _ in range(max(plan) + 1)]
    for t in range(len(numels) - 1, -1, -1):
        buckets[plan[t]].append(t)
    return numels, offs, buckets


def _vit_step(comm, grads, w, v, numels, offs, buckets):
    for b in buckets:
        ts = [[g[offs[t]:offs[t + 1]] for g in grads] for t in b]
        gar.ar_bucket_all_reduce(comm, ts, [numels[t] for t in b], gar.AR_BF16, gar.AR_MEAN,
                                 sgd=(0.1, 0.9, [w[offs[t]:offs[t + 1]] for t in b],
                                      [v[offs[t]:offs[t + 1]] for t in b], 1))


def test_vit_b16_bucketed_sgd_full_size_sampled(path):
    """ViT-B/16: 86,567,656 bf16 gradients per replica ~N(0, 1e-3) (replica
    r from seed 100 + r), P=8, 8 buckets of <= 25 MiB in reverse order,
    Mean fused with SGD (momentum 0.9, lr 0.1) on fp32 master weights
    ~N(0, 0.02) (seed 200), write-back on; two steps.  Sampled outputs
    (every tensor's first and last element plus 200,000 random positions)
    equal the oracle's bits; every replica holds the same gradient."""
    P = 8
    numels, offs, buckets = _vit_buckets(25 << 20)
    assert len(buckets) == 8
    n = int(offs[-1])
    assert n == workloads.VIT_B16_PARAMS
    grads = replicas(P, n, "bf16", "normal", workloads.VIT_GRAD_SEED, std=workloads.VIT_GRAD_STD)
    w = empty(n, "f32")
    wgpu.fill(w, "normal", workloads.VIT_MASTER_SEED, std=workloads.VIT_MASTER_STD)
    v = torch.zeros(n, dtype=torch.float32, device=dev())
    idx = sample_indices(n, 200_000, 3, extra=[int(o) for o in offs[1:-1]] +
                         [int(o) - 1 for o in offs[1:]])
    cols = host_replicas(P, 0, "bf16", "normal", workloads.VIT_GRAD_SEED,
                         std=workloads.VIT_GRAD_STD, idx=idx)
    hw = workloads.normal_f32(workloads.VIT_MASTER_SEED, 0, std=workloads.VIT_MASTER_STD, idx=idx)
    hv = np.zeros(idx.size, np.float32)
    comm = init(P, gar.AR_MEAN, path)
    try:
        for step in range(2):
            _vit_step(comm, grads, w, v, numels, offs, buckets)
            torch.cuda.synchronize()
            assert gar.ar_get_async_error(comm) == gar.AR_OK
            oracle.bucket_all_reduce([cols], op=oracle.MEAN, sgd=(0.1, 0.9, [hw], [hv], 1))
            assert_bits_equal(gather(w, idx), hw, f"step {step} master")
            assert_bits_equal(gather(v, idx), hv, f"step {step} momentum")
            for r in (0, 3, P - 1):
                assert_bits_equal(gather(grads[r], idx), cols[r], f"step {step} grad {r}")
            for r in range(1, P):
                assert bits_equal_device(grads[r], grads[0]), r
    finally:
        gar.ar_destroy(comm)


def test_vit_b16_step_as_benchmarked():
    """The ViT-B/16 step exactly as bench.py times it: its own VitStep
    object (the same buffers, seeds and prepared calls), two steps through
    the reducer (marks in reverse order, buckets on two streams), then one
    step of the same 8 bucket calls back to back on one stream.  Sampled
    outputs equal three oracle steps bit for bit; every replica holds the
    same gradient."""
    import bench
    P = bench.P_VIT
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    vs = None
    try:
        vs = bench.VitStep(comm, dev())
        n = vs.n
        assert n == workloads.VIT_B16_PARAMS and len(vs.calls) == 8
        idx = sample_indices(n, 200_000, 5, extra=[int(o) for o in vs.offs[1:-1]] +
                             [int(o) - 1 for o in vs.offs[1:]])
        cols = host_replicas(P, 0, "bf16", "normal", workloads.VIT_GRAD_SEED,
                             std=workloads.VIT_GRAD_STD, idx=idx)
        hw = workloads.normal_f32(workloads.VIT_MASTER_SEED, 0, std=workloads.VIT_MASTER_STD,
                                  idx=idx)
        hv = np.zeros(idx.size, np.float32)
        stream = torch.cuda.Stream(dev())
        for step, run in enumerate((vs.step, vs.step, vs.step_serial)):
            with torch.cuda.stream(stream):
                run(stream)
            torch.cuda.synchronize()
            assert gar.ar_get_async_error(comm) == gar.AR_OK
            oracle.bucket_all_reduce([cols], op=oracle.MEAN, sgd=(0.1, 0.9, [hw], [hv], 1))
            assert_bits_equal(gather(vs.w, idx), hw, f"step {step} master")
            assert_bits_equal(gather(vs.v, idx), hv, f"step {step} momentum")
            for r in (0, 5, P - 1):
                assert_bits_equal(gather(vs.grads[r], idx), cols[r], f"step {step} grad {r}")
            for r in range(1, P):
                assert bits_equal_device(vs.grads[r], vs.grads[0]), r
    finally:
        if vs is not None:
            vs.close()
        gar.ar_destroy(comm)


def test_vit_b16_e2e_pipelined_steps():
    """The end-to-end step bench.py times (E2EStep): gradients copied in
    from pinned host memory bucket by bucket, the reducer, the updated
    weights copied out, consecutive steps ordered per bucket only.  After
    four steps issued back to back, the weights copied to the host and the
    gradient replicas equal four oracle steps (each on the original
    gradients, which every step copies in afresh), sampled bit for bit: no
    copy-in overtook a kernel that still read its bucket, and no kernel
    overtook a copy-out."""
    import bench
    P = bench.P_VIT
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    vs = None
    try:
        vs = bench.VitStep(comm, dev())
        e2e = bench.E2EStep(vs, dev())
        n = vs.n
        idx = sample_indices(n, 200_000, 6, extra=[int(o) for o in vs.offs[1:-1]] +
                             [int(o) - 1 for o in vs.offs[1:]])
        cols0 = host_replicas(P, 0, "bf16", "normal", workloads.VIT_GRAD_SEED,
                              std=workloads.VIT_GRAD_STD, idx=idx)
        hw = workloads.normal_f32(workloads.VIT_MASTER_SEED, 0, std=workloads.VIT_MASTER_STD,
                                  idx=idx)
        hv = np.zeros(idx.size, np.float32)
        stream = torch.cuda.Stream(dev())
        with torch.cuda.stream(stream):
            e2e.start(stream)
            for _ in range(4):
                e2e.step(stream)
            e2e.finish(stream)
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
        for _ in range(4):
            cols = [c.copy() for c in cols0]
            oracle.bucket_all_reduce([cols], op=oracle.MEAN, sgd=(0.1, 0.9, [hw], [hv], 1))
        it = torch.from_numpy(idx.astype(np.int64))
        assert_bits_equal(e2e.host_w[it].numpy(), hw, "weights copied out")
        assert_bits_equal(gather(vs.v, idx), hv, "momentum")
        for r in (0, 4, P - 1):
            assert_bits_equal(gather(vs.grads[r], idx), cols[r], f"grad {r}")
    finally:
        if vs is not None:
            vs.close()
        gar.ar_destroy(comm)


def test_vit_small_cap_full_check(path):
    """The same step with 4 MiB buckets (many more, smaller launches) on the
    first 12,000,000 ViT elements, checked against the oracle on every
    element."""
    P = 8
    numels, offs, _ = _vit_buckets(4 << 20)
    keep = int(np.searchsorted(offs, 12_000_000))
    numels = numels[:keep]
    offs = offs[:keep + 1]
    plan = gar.ar_bucket_plan([2 * k for k in numels], 4 << 20)
    buckets = [[] for _ in range(max(plan) + 1)]
    for t in range(len(numels) - 1, -1, -1):
        buckets[plan[t]].append(t)
    n = int(offs[-1])
    grads = replicas(P, n, "bf16", "normal", 100, std=1e-3)
    w = empty(n, "f32")
    wgpu.fill(w, "normal", 200, std=0.02)
    v = torch.zeros(n, dtype=torch.float32, device=dev())
    comm = init(P, gar.AR_MEAN, path)
    try:
        _vit_step(comm, grads, w, v, numels, offs, buckets)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    host = host_replicas(P, n, "bf16", "normal", 100, std=1e-3)
    hw = [workloads.normal_f32(200, n, std=0.02)]
    hv = [np.zeros(n, np.float32)]
    oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
    assert_bits_equal(to_np(w), hw[0], "master")
    assert_bits_equal(to_np(v), hv[0], "momentum")
    for r in (0, P - 1):
        assert_bits_equal(to_np(grads[r]), host[r], f"grad {r}")


def test_large_bucket_rs_ag_ar(path):
    """P=4 replicas of 2**30 fp32 ~N(0,1) (4 GiB each): reduce-scatter then
    all-gather equals the fused all-reduce (Sum) bit for bit on the device;
    sampled outputs equal the oracle's."""
    P, n = 4, 1 << 30
    shard = n // P
    xs = replicas(P, n, "f32", "normal", 0)
    comm = init(P, gar.AR_SUM, path)
    try:
        ar = [empty(n, "f32") for _ in range(P)]
        gar.ar_all_reduce(comm, xs, ar, n, gar.AR_F32, gar.AR_SUM)
        rs = [empty(shard, "f32") for _ in range(P)]
        gar.ar_reduce_scatter(comm, xs, rs, n, gar.AR_F32, gar.AR_SUM)
        torch.cuda.synchronize()
        idx = sample_indices(n, 100_000, 4, extra=[shard - 1, shard, 3 * shard])
        want = oracle.all_reduce(host_replicas(P, 0, "f32", "normal", 0, idx=idx), op=oracle.SUM)
        for r in range(P):
            assert_bits_equal(gather(ar[r], idx), want[r], f"AR {r}")
        for r in range(P):
            sel = (idx >= r * shard) & (idx < (r + 1) * shard)
            assert_bits_equal(gather(rs[r], idx[sel] - r * shard), want[0][sel], f"RS {r}")
        del xs
        ag = [empty(n, "f32") for _ in range(P)]
        gar.ar_all_gather(comm, rs, ag, n, gar.AR_F32)
        torch.cuda.synchronize()
        for r in range(P):
            assert bits_equal_device(ag[r], ar[r]), r
    finally:
        gar.ar_destroy(comm)


SWEEP_BYTES = [4096 * 4 ** k for k in range(10)]   # 4 KiB .. 1 GiB per replica


@pytest.mark.parametrize("P", [2, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_sweep(path, P, dt):
    """Every size of the sweep, Sum and Mean, in place, plus a broadcast
    from rank 0: full oracle check up to 4 MiB per replica, sampled above."""
    s = 4 if dt == "f32" else 2
    comm = init(P, gar.AR_MEAN, path)
    try:
        for nbytes in SWEEP_BYTES:
            n = nbytes // s
            for op in ("sum", "mean"):
                xs = replicas(P, n, dt, "uniform", 0)
                gar.ar_all_reduce(comm, xs, xs, n, DT[dt], OP[op])
                torch.cuda.synchronize()
                if nbytes <= 4 << 20:
                    want = oracle.all_reduce(host_replicas(P, n, dt, "uniform", 0),
                                             op=ORACLE_OP[op])
                    for r in (0, P - 1):
                        assert_bits_equal(to_np(xs[r]), want[r], f"{nbytes} {op} {r}")
                else:
                    idx = sample_indices(n, 20_000, nbytes)
                    want = oracle.all_reduce(host_replicas(P, 0, dt, "uniform", 0, idx=idx),
                                             op=ORACLE_OP[op])
                    for r in (0, P - 1):
                        assert_bits_equal(gather(xs[r], idx), want[r], f"{nbytes} {op} {r}")
                    for r in range(1, P):
                        assert bits_equal_device(xs[r], xs[0]), (nbytes, op, r)
                del xs
            xs = replicas(P, n, dt, "uniform", 0)
            gar.ar_broadcast(comm, xs, n, DT[dt], 0)
            torch.cuda.synchronize()
            root = replicas(1, n, dt, "uniform", 0)[0]
            for r in range(P):
                assert bits_equal_device(xs[r], root), (nbytes, r)
            del xs, root
    finally:
        gar.ar_destroy(comm)
