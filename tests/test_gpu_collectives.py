"""GPU parity of the flat collectives through the C ABI against the CPU
oracle: all-reduce (Sum/Mean, fp32/bf16, in and out of place), reduce-scatter,
all-gather and broadcast, over P = 1..16, sizes that are empty, tiny, ragged
and several tiles long, and buffers that are not 16-byte aligned.  Every
comparison is bit for bit."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
from gpucase import (DT, OP, ORACLE_OP, PATHS, assert_bits_equal, bits_equal_device, dev, empty,
                     host_replicas, init, replicas, to_np)

pytestmark = pytest.mark.gpu

SIZES = (0, 1, 3, 17, 4097, 200_003)


@pytest.fixture(scope="module", params=PATHS)
def comms(request):
    """Comms per P, with the reduce kernel of this run's path."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    made = {}

    def get(P):
        if P not in made:
            made[P] = init(P, gar.AR_MEAN, request.param)
        return made[P]

    yield get
    for c in made.values():
        gar.ar_destroy(c)


def _sync_ok(comm):
    torch.cuda.synchronize()
    assert gar.ar_get_async_error(comm) == gar.AR_OK


def test_tiny_config_mean_in_place(comms):
    """P=4 replicas of 1,048,576 fp32 U(-1,1) elements (replica r from seed
    r), Mean, in place: every replica equals the oracle bit for bit."""
    P, n = 4, 1 << 20
    xs = replicas(P, n, "f32", "uniform", 0)
    comm = comms(P)
    gar.ar_all_reduce(comm, xs, xs, n, gar.AR_F32, gar.AR_MEAN)
    _sync_ok(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "uniform", 0), op=oracle.MEAN)
    for r in range(P):
        assert_bits_equal(to_np(xs[r]), want[r], f"replica {r}")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 12, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["sum", "mean"])
@pytest.mark.parametrize("n", SIZES)
def test_all_reduce_out_of_place(comms, P, dt, op, n):
    xs = replicas(P, n, dt, "normal", 10 * P)
    ys = [empty(n, dt) for _ in range(P)]
    comm = comms(P)
    gar.ar_all_reduce(comm, xs, ys, n, DT[dt], OP[op])
    _sync_ok(comm)
    host = host_replicas(P, n, dt, "normal", 10 * P)
    want = oracle.all_reduce(host, op=ORACLE_OP[op])
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"recv {r}")
        assert_bits_equal(to_np(xs[r]), host[r], f"send {r} untouched")


@pytest.mark.parametrize("P", [2, 4, 7, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_all_reduce_unaligned_and_in_place(comms, P, dt):
    """Buffers one element past a 16-byte boundary take the scalar path;
    in place and out of place give the oracle's bits."""
    n = 50_021
    comm = comms(P)
    host = host_replicas(P, n, dt, "uniform", 3)
    want = oracle.all_reduce(host, op=oracle.MEAN)
    xs = replicas(P, n, dt, "uniform", 3, offset=1)
    gar.ar_all_reduce(comm, xs, xs, n, DT[dt], gar.AR_MEAN)
    _sync_ok(comm)
    for r in range(P):
        assert_bits_equal(to_np(xs[r]), want[r], f"unaligned in place {r}")
    xs = replicas(P, n, dt, "uniform", 3)
    ys = [empty(n, dt, offset=1) for _ in range(P)]
    gar.ar_all_reduce(comm, xs, ys, n, DT[dt], gar.AR_MEAN)
    _sync_ok(comm)
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"unaligned recv {r}")


def test_default_op_and_side_stream(comms):
    """AR_OP_DEFAULT takes the comm's Mean; work runs on the given stream."""
    P, n = 4, 70_001
    comm = comms(P)
    xs = replicas(P, n, "f32", "uniform", 5)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gar.ar_all_reduce(comm, xs, xs, n, gar.AR_F32, gar.AR_OP_DEFAULT, stream=s)
    s.synchronize()
    want = oracle.all_reduce(host_replicas(P, n, "f32", "uniform", 5), op=oracle.MEAN)
    assert_bits_equal(to_np(xs[2]), want[2], "default op")


def test_special_values(comms):
    """Signed zeros, infinities, subnormals and values that overflow: the
    GPU gives the oracle's bits; NaN results are NaN in both."""
    P = 4
    vals = np.array([-0.0, 0.0, 1e-45, -1e-45, 1e-40, 3e38, np.inf, -np.inf, 1.0, 5e-39],
                    np.float32)
    host = [np.roll(vals, r).copy() for r in range(P)]
    host[0][0] = -0.0
    host[1][0] = -0.0
    host[2][0] = -0.0
    host[3][0] = -0.0
    comm = comms(P)
    for dt in ("f32", "bf16"):
        h = host if dt == "f32" else [(x.view(np.uint32) >> 16).astype(np.uint16) for x in host]
        xs = [torch.from_numpy(x.view(np.int16) if dt == "bf16" else x).to(dev()) for x in h]
        if dt == "bf16":
            xs = [x.view(torch.bfloat16) for x in xs]
        for op in ("sum", "mean"):
            ys = [torch.empty_like(x) for x in xs]
            gar.ar_all_reduce(comm, xs, ys, vals.size, DT[dt], OP[op])
            _sync_ok(comm)
            want = oracle.all_reduce(h, op=ORACLE_OP[op])
            got = to_np(ys[0])
            wf = want[0] if dt == "f32" else (want[0].astype(np.uint32) << 16).view(np.float32)
            gf = got if dt == "f32" else (got.astype(np.uint32) << 16).view(np.float32)
            nan = np.isnan(wf)
            assert np.array_equal(nan, np.isnan(gf)), (dt, op)
            assert_bits_equal(got[~nan], want[0][~nan], f"{dt} {op}")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 10, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shard", [0, 1, 5, 4096, 33_331])
def test_reduce_scatter(comms, P, dt, shard):
    n = shard * P
    comm = comms(P)
    host = host_replicas(P, n, dt, "normal", 40)
    for op in ("sum", "mean"):
        want = oracle.reduce_scatter(host, op=ORACLE_OP[op])
        xs = replicas(P, n, dt, "normal", 40)
        ys = [empty(shard, dt) for _ in range(P)]
        gar.ar_reduce_scatter(comm, xs, ys, n, DT[dt], OP[op])
        _sync_ok(comm)
        for r in range(P):
            assert_bits_equal(to_np(ys[r]), want[r], f"out of place {op} {r}")
        # in place: rank r's shard lands in its own buffer at offset r*shard
        xs = replicas(P, n, dt, "normal", 40)
        ys = [x[r * shard:(r + 1) * shard] for r, x in enumerate(xs)]
        gar.ar_reduce_scatter(comm, xs, ys, n, DT[dt], OP[op])
        _sync_ok(comm)
        for r in range(P):
            assert_bits_equal(to_np(ys[r]), want[r], f"in place {op} {r}")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shard", [0, 1, 5, 4096, 33_331])
def test_all_gather(comms, P, dt, shard):
    n = shard * P
    comm = comms(P)
    host = host_replicas(P, shard, dt, "uniform", 50)
    want = oracle.all_gather(host)
    xs = replicas(P, shard, dt, "uniform", 50)
    ys = [empty(n, dt) for _ in range(P)]
    gar.ar_all_gather(comm, xs, ys, n, DT[dt])
    _sync_ok(comm)
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"out of place {r}")
    # in place: rank r's contribution already sits at offset r*shard of recv[r]
    ys = [empty(n, dt) for _ in range(P)]
    for r in range(P):
        ys[r][r * shard:(r + 1) * shard].copy_(xs[r])
    gar.ar_all_gather(comm, [y[r * shard:(r + 1) * shard] for r, y in enumerate(ys)], ys, n,
                      DT[dt])
    _sync_ok(comm)
    for r in range(P):
        assert_bits_equal(to_np(ys[r]), want[r], f"in place {r}")


@pytest.mark.parametrize("P", [1, 2, 5, 8, 16])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("n", [0, 1, 9, 200_003])
def test_broadcast(comms, P, dt, n):
    comm = comms(P)
    for root in sorted({0, P - 1, P // 2}):
        xs = replicas(P, n, dt, "uniform", 60)
        host = host_replicas(P, n, dt, "uniform", 60)
        gar.ar_broadcast(comm, xs, n, DT[dt], root)
        _sync_ok(comm)
        want = oracle.broadcast(host, root=root)
        for r in range(P):
            assert_bits_equal(to_np(xs[r]), want[r], f"root {root} rank {r}")


@pytest.mark.parametrize("P", [2, 3, 4, 8])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_rs_then_ag_equals_all_reduce_on_gpu(comms, P, dt):
    """Invariant on the device: all-gather(reduce-scatter(x)) == all-reduce(x)."""
    shard = 123_457
    n = shard * P
    comm = comms(P)
    xs = replicas(P, n, dt, "normal", 70)
    ar = [empty(n, dt) for _ in range(P)]
    gar.ar_all_reduce(comm, xs, ar, n, DT[dt], gar.AR_SUM)
    rs = [empty(shard, dt) for _ in range(P)]
    gar.ar_reduce_scatter(comm, xs, rs, n, DT[dt], gar.AR_SUM)
    ag = [empty(n, dt) for _ in range(P)]
    gar.ar_all_gather(comm, rs, ag, n, DT[dt])
    _sync_ok(comm)
    for r in range(P):
        assert bits_equal_device(ag[r], ar[r]), r


def test_invalid_arguments_enqueue_nothing(comms):
    """Wrong calls are refused on the host with AR_ERR_INVALID_ARG (or
    AR_ERR_STATE) before any launch; the buffers stay untouched."""
    P, n = 4, 1000
    comm = comms(P)
    xs = replicas(P, n, "f32", "uniform", 80)
    before = [to_np(x).copy() for x in xs]

    def refused(fn, *a, status=gar.AR_ERR_INVALID_ARG):
        with pytest.raises(gar.GarError) as e:
            fn(*a)
        assert e.value.status == status

    ys = [empty(n, "f32") for _ in range(P)]
    refused(gar.ar_all_reduce, comm, xs, [ys[0], ys[0], ys[2], ys[3]], n, gar.AR_F32, gar.AR_SUM)
    refused(gar.ar_all_reduce, comm, xs, [xs[1], ys[1], ys[2], ys[3]], n, gar.AR_F32, gar.AR_SUM)
    refused(gar.ar_all_reduce, comm, xs, ys, n, 7, gar.AR_SUM)
    refused(gar.ar_all_reduce, comm, xs, ys, n, gar.AR_F32, 5)
    refused(gar.ar_all_reduce, comm, [xs[0].data_ptr() + 2] + xs[1:], ys, n - 1, gar.AR_F32,
            gar.AR_SUM)                                           # not element aligned
    refused(gar.ar_all_reduce, comm, xs, ys, n + 10 ** 9, gar.AR_F32, gar.AR_SUM)  # past the end
    host = np.zeros(n, np.float32)
    refused(gar.ar_all_reduce, comm, [host.ctypes.data] + xs[1:], ys, n, gar.AR_F32,
            gar.AR_SUM)                                           # pageable host memory
    refused(gar.ar_reduce_scatter, comm, xs, [y[:n // P] for y in ys], n - 1, gar.AR_F32,
            gar.AR_SUM)                                           # count % P != 0
    refused(gar.ar_broadcast, comm, xs, n, gar.AR_F32, P)          # root out of range
    refused(gar.ar_broadcast, comm, [xs[0], xs[0], xs[2], xs[3]], n, gar.AR_F32, 0)
    refused(gar.ar_all_reduce, 12345, xs, ys, n, gar.AR_F32, gar.AR_SUM, status=gar.AR_ERR_STATE)
    torch.cuda.synchronize()
    for r in range(P):
        assert_bits_equal(to_np(xs[r]), before[r], "untouched")
    c = gar.ar_init(2, 0, gar.AR_SUM)
    gar.ar_destroy(c)
    refused(gar.ar_destroy, c, status=gar.AR_ERR_STATE)
    refused(gar.ar_init, 0, 0, gar.AR_SUM)
    refused(gar.ar_init, 17, 0, gar.AR_SUM)
    refused(gar.ar_init, 2, 9999, gar.AR_SUM)


def test_device_generator_matches_host():
    """The device-side input generator reproduces the host's bits."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    for dt in ("f32", "bf16"):
        for kind, std in (("uniform", 1.0), ("normal", 1e-3), ("normal", 0.02)):
            t = replicas(1, 100_003, dt, kind, 7, std=std)[0]
            assert_bits_equal(to_np(t), host_replicas(1, 100_003, dt, kind, 7, std=std)[0],
                              f"{dt} {kind}")


def test_prepared_calls_match_direct_calls(comms):
    """PreparedCall (arguments marshalled once) gives the direct call's bits,
    and a CUDA graph of it replays the same computation."""
    P, n = 8, 100_003
    comm = comms(P)
    xs = replicas(P, n, "f32", "uniform", 90)
    ys = [empty(n, "f32") for _ in range(P)]
    zs = [empty(n, "f32") for _ in range(P)]
    gar.ar_all_reduce(comm, xs, ys, n, gar.AR_F32, gar.AR_MEAN)
    call = gar.PreparedCall("ar_all_reduce", comm, xs, zs, n, gar.AR_F32, gar.AR_MEAN)
    call()
    _sync_ok(comm)
    for r in range(P):
        assert bits_equal_device(ys[r], zs[r]), r
    for z in zs:
        z.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    call(side)
    torch.cuda.synchronize()
    for z in zs:
        z.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    for r in range(P):
        assert bits_equal_device(ys[r], zs[r]), r
    bc = gar.PreparedCall("ar_broadcast", comm, zs, n, gar.AR_F32, 3)
    bc()
    torch.cuda.synchronize()
    assert bits_equal_device(zs[0], zs[3])


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_chained_collectives_without_syncs(comms, dt):
    """24 collectives of every kind on the same buffers, issued back to back
    on one stream with no synchronisation in between (each kernel may start
    while the previous one drains, under programmatic dependent launch):
    all-reduce Sum and Mean in and out of place, reduce-scatter and
    all-gather in place, broadcast from a random root, and the bucketed
    Mean + SGD step.  The result equals the oracle running the same
    sequence, bit for bit.  Shards of 65,541 elements leave most of them off
    16-byte boundaries, so both access paths take part."""
    P, s = 4, 65_541
    n = P * s
    h = n // 2
    comm = comms(P)
    xs = replicas(P, n, dt, "uniform", 90)
    ys = [empty(n, dt) for _ in range(P)]
    w = torch.zeros(n, dtype=torch.float32, device=dev())
    v = torch.zeros(n, dtype=torch.float32, device=dev())
    hx = host_replicas(P, n, dt, "uniform", 90)
    hy = [None] * P
    hw = np.zeros(n, np.float32)
    hv = np.zeros(n, np.float32)
    rng = np.random.default_rng(91)
    kinds = ["ar_sum", "ar_mean", "ar_to_y", "ar_from_y", "rs", "ag", "bc", "bucket_sgd"]
    seq = [kinds[int(k)] for k in rng.integers(0, len(kinds), 24)]
    seq[:3] = ["ar_to_y", "rs", "ag"]          # ys is written before any op reads it
    t = DT[dt]
    for k, op in enumerate(seq):
        if op == "ar_sum":
            gar.ar_all_reduce(comm, xs, xs, n, t, gar.AR_SUM)
            hx = oracle.all_reduce(hx, op=oracle.SUM)
        elif op == "ar_mean":
            gar.ar_all_reduce(comm, xs, xs, n, t, gar.AR_MEAN)
            hx = oracle.all_reduce(hx, op=oracle.MEAN)
        elif op == "ar_to_y":
            gar.ar_all_reduce(comm, xs, ys, n, t, gar.AR_MEAN)
            hy = oracle.all_reduce(hx, op=oracle.MEAN)
        elif op == "ar_from_y":
            gar.ar_all_reduce(comm, ys, xs, n, t, gar.AR_SUM)
            hx = oracle.all_reduce(hy, op=oracle.SUM)
        elif op == "rs":
            gar.ar_reduce_scatter(comm, xs, [x[r * s:(r + 1) * s] for r, x in enumerate(xs)], n, t,
                                  gar.AR_MEAN)
            shards = oracle.reduce_scatter(hx, op=oracle.MEAN)
            for r in range(P):
                hx[r][r * s:(r + 1) * s] = shards[r]
        elif op == "ag":
            gar.ar_all_gather(comm, [x[r * s:(r + 1) * s] for r, x in enumerate(xs)], xs, n, t)
            hx = oracle.all_gather([hx[r][r * s:(r + 1) * s].copy() for r in range(P)])
        elif op == "bc":
            root = int(rng.integers(0, P))
            gar.ar_broadcast(comm, xs, n, t, root)
            oracle.broadcast(hx, root=root)
        else:
            gar.ar_bucket_all_reduce(comm, [[x[:h] for x in xs], [x[h:] for x in xs]], [h, n - h],
                                     t, gar.AR_MEAN,
                                     sgd=(0.1, 0.9, [w[:h], w[h:]], [v[:h], v[h:]], 1))
            tens = [[hx[r][:h].copy() for r in range(P)], [hx[r][h:].copy() for r in range(P)]]
            ws, vs = [hw[:h].copy(), hw[h:].copy()], [hv[:h].copy(), hv[h:].copy()]
            oracle.bucket_all_reduce(tens, op=oracle.MEAN, sgd=(0.1, 0.9, ws, vs, 1))
            hx = [np.concatenate([tens[0][r], tens[1][r]]) for r in range(P)]
            hw, hv = np.concatenate(ws), np.concatenate(vs)
    _sync_ok(comm)
    for r in range(P):
        got, want = to_np(xs[r]), hx[r]
        wf = want.astype(np.float32) if dt == "f32" else (want.astype(np.uint32) << 16).view(np.float32)
        assert not np.isnan(wf).any()
        assert_bits_equal(got, want, f"{dt} replica {r} after {seq}")
    assert_bits_equal(to_np(w), hw, "master")
    assert_bits_equal(to_np(v), hv, "momentum")


def _copy_comm(P, group):
    """A comm whose windowed copies take `group` destinations per item
    (None: the library's default rule)."""
    import os
    old = os.environ.get("GAR_COPY_GROUP")
    if group is not None:
        os.environ["GAR_COPY_GROUP"] = str(group)
    try:
        return gar.ar_init(P, 0, gar.AR_MEAN)
    finally:
        if old is None:
            os.environ.pop("GAR_COPY_GROUP", None)
        else:
            os.environ["GAR_COPY_GROUP"] = old


# Sizes above the 32 MB of source at which copies take the windowed order:
# a ragged tail (not a whole number of 16-byte vectors) and a partial last
# window.
WINDOWED_BYTES = (32 << 20) + (3 << 20) + 6


@pytest.mark.parametrize("P", [2, 3, 5, 8])
@pytest.mark.parametrize("group", [None, 1, 2, 3, 7])
def test_windowed_all_gather(P, group):
    """All-gather of shards large enough for the windowed order, with every
    destination-group size: out of place, in place, in place for some ranks
    only (segments with different destination counts), and shards one
    element past a 16-byte boundary (the scalar path), against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dt = "bf16"
    shard = WINDOWED_BYTES // 2 // P
    n = shard * P
    comm = _copy_comm(P, group)
    try:
        host = host_replicas(P, shard, dt, "uniform", 80 + P)
        want = oracle.all_gather(host)
        xs = replicas(P, shard, dt, "uniform", 80 + P)
        ys = [empty(n, dt) for _ in range(P)]
        gar.ar_all_gather(comm, xs, ys, n, DT[dt])
        _sync_ok(comm)
        for r in range(P):
            assert_bits_equal(to_np(ys[r]), want[r], f"out of place {r}")
        for in_place in ({*range(P)}, {r for r in range(P) if r % 2 == 0}):
            ys = [empty(n, dt) for _ in range(P)]
            send = []
            for r in range(P):
                if r in in_place:
                    ys[r][r * shard:(r + 1) * shard].copy_(xs[r])
                    send.append(ys[r][r * shard:(r + 1) * shard])
                else:
                    send.append(xs[r])
            gar.ar_all_gather(comm, send, ys, n, DT[dt])
            _sync_ok(comm)
            for r in range(P):
                assert_bits_equal(to_np(ys[r]), want[r], f"in place {sorted(in_place)} rank {r}")
        xs1 = replicas(P, shard, dt, "uniform", 80 + P, offset=1)
        ys1 = [empty(n, dt, offset=1) for _ in range(P)]
        gar.ar_all_gather(comm, xs1, ys1, n, DT[dt])
        _sync_ok(comm)
        for r in range(P):
            assert_bits_equal(to_np(ys1[r]), want[r], f"unaligned {r}")
    finally:
        gar.ar_destroy(comm)


@pytest.mark.parametrize("P", [2, 4, 8, 16])
@pytest.mark.parametrize("group", [None, 1, 3, 15])
def test_windowed_broadcast(P, group):
    """Broadcast of a buffer large enough for the windowed order, from the
    first, a middle and the last root, aligned and unaligned, against the
    oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dt = "f32"
    n = WINDOWED_BYTES // 4 + 1
    comm = _copy_comm(P, group)
    try:
        for root, offset in ((0, 0), (P // 2, 1), (P - 1, 0)):
            xs = replicas(P, n, dt, "uniform", 90, offset=offset)
            gar.ar_broadcast(comm, xs, n, DT[dt], root)
            _sync_ok(comm)
            want = host_replicas(1, n, dt, "uniform", 90 + root)[0]   # the root's draws
            for r in range(P):
                assert_bits_equal(to_np(xs[r]), want, f"root {root} rank {r}")
    finally:
        gar.ar_destroy(comm)


# Between 8 MiB and 32 MB of source a copy takes two vectors per thread in the
# classic order; below 8 MiB one.
MID_BYTES = (12 << 20) + 6


@pytest.mark.parametrize("P", [2, 3, 8])
@pytest.mark.parametrize("nbytes", [MID_BYTES, (6 << 20) + 2])
def test_mid_size_copies(P, nbytes):
    """All-gather (out of place, in place, in place for some ranks,
    unaligned) and broadcast (three roots, unaligned) at sizes of each
    small-copy tile class, against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dt = "bf16"
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        shard = nbytes // 2 // P
        n = shard * P
        host = host_replicas(P, shard, dt, "uniform", 110 + P)
        want = oracle.all_gather(host)
        xs = replicas(P, shard, dt, "uniform", 110 + P)
        for in_place in (set(), {*range(P)}, {r for r in range(P) if r % 2 == 1}):
            ys = [empty(n, dt) for _ in range(P)]
            send = []
            for r in range(P):
                if r in in_place:
                    ys[r][r * shard:(r + 1) * shard].copy_(xs[r])
                    send.append(ys[r][r * shard:(r + 1) * shard])
                else:
                    send.append(xs[r])
            gar.ar_all_gather(comm, send, ys, n, DT[dt])
            _sync_ok(comm)
            for r in range(P):
                assert_bits_equal(to_np(ys[r]), want[r], f"in place {sorted(in_place)} rank {r}")
        xs1 = replicas(P, shard, dt, "uniform", 110 + P, offset=1)
        ys1 = [empty(n, dt, offset=1) for _ in range(P)]
        gar.ar_all_gather(comm, xs1, ys1, n, DT[dt])
        _sync_ok(comm)
        for r in range(P):
            assert_bits_equal(to_np(ys1[r]), want[r], f"unaligned {r}")
        nb = nbytes // 2
        for root, offset in ((0, 1), (P - 1, 0)):
            bs = replicas(P, nb, dt, "uniform", 120, offset=offset)
            gar.ar_broadcast(comm, bs, nb, DT[dt], root)
            _sync_ok(comm)
            src = host_replicas(1, nb, dt, "uniform", 120 + root)[0]
            for r in range(P):
                assert_bits_equal(to_np(bs[r]), src, f"broadcast root {root} rank {r}")
    finally:
        gar.ar_destroy(comm)
