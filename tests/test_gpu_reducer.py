"""The DDP gradient reducer (ar_reducer_*) on the GPU, against the CPU
oracle: buckets planned in reverse order, launched as their last gradient is
marked ready, on two communication streams ordered after the streams that
produced the gradients; results identical to the per-bucket collective."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import PATHS, assert_bits_equal, dev, empty, host_replicas, init, to_np
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _vit_prefix(n_target):
    numels = workloads.vit_b16_numels()
    offs = np.concatenate([[0], np.cumsum(numels)])
    keep = int(np.searchsorted(offs, n_target))
    return numels[:keep], offs[:keep + 1]


def _setup(P, numels, offs, dt="bf16", seed=100):
    n = int(offs[-1])
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    flat = [torch.empty(n, dtype=tdt, device=dev()) for _ in range(P)]
    for r, g in enumerate(flat):
        wgpu.fill(g, "normal", seed + r, std=1e-3)
    w = torch.empty(n, dtype=torch.float32, device=dev())
    wgpu.fill(w, "normal", 200, std=0.02)
    v = torch.zeros(n, dtype=torch.float32, device=dev())
    grads = [[g[offs[t]:offs[t + 1]] for g in flat] for t in range(len(numels))]
    ws = [w[offs[t]:offs[t + 1]] for t in range(len(numels))]
    vs = [v[offs[t]:offs[t + 1]] for t in range(len(numels))]
    return flat, w, v, grads, ws, vs


@pytest.mark.parametrize("path", PATHS)
def test_reducer_two_steps_match_oracle(path):
    """12M elements of the ViT-B/16 set, 4 MiB buckets, Mean + SGD, two
    steps with every tensor marked in reverse order on the current stream."""
    P = 8
    numels, offs = _vit_prefix(12_000_000)
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs)
    comm = init(P, gar.AR_MEAN, path)
    red = gar.Reducer(comm, grads, numels, gar.AR_BF16, 4 << 20, gar.AR_MEAN,
                      sgd=(0.1, 0.9, ws, vs, 1))
    try:
        assert red.bucket_of() == gar.ar_bucket_plan([2 * k for k in numels], 4 << 20)
        host = host_replicas(P, n, "bf16", "normal", 100, std=1e-3)
        hw = [workloads.normal_f32(200, n, std=0.02)]
        hv = [np.zeros(n, np.float32)]
        for step in range(2):
            for t in range(len(numels) - 1, -1, -1):
                red.mark_ready(t)
            red.finalize()
            torch.cuda.synchronize()
            oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
            assert_bits_equal(to_np(w), hw[0], f"step {step} master")
            assert_bits_equal(to_np(v), hv[0], f"step {step} momentum")
            for r in (0, P - 1):
                assert_bits_equal(to_np(flat[r]), host[r], f"step {step} grad {r}")
    finally:
        red.destroy()
        gar.ar_destroy(comm)


@pytest.mark.parametrize("P", [3, 6, 12])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_reducer_runtime_p_combined_launch_matches_oracle(P, dt):
    """A rank count that is not a power of two (the kernels sized for up to
    4, 8 or 12 ranks, and the Mean's division): 4M elements of the ViT-B/16
    set, 2 MiB buckets, Mean + SGD, every tensor marked in one
    mark_ready_many call (so the buckets go out as combined launches), two
    steps."""
    numels, offs = _vit_prefix(4_000_000)
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    red = gar.Reducer(comm, grads, numels, gar.AR_BF16 if dt == "bf16" else gar.AR_F32, 2 << 20,
                      gar.AR_MEAN, sgd=(0.1, 0.9, ws, vs, 1))
    try:
        host = host_replicas(P, n, dt, "normal", 100, std=1e-3)
        hw = [workloads.normal_f32(200, n, std=0.02)]
        hv = [np.zeros(n, np.float32)]
        for step in range(2):
            red.mark_ready_many(list(range(len(numels) - 1, -1, -1)))
            red.finalize()
            torch.cuda.synchronize()
            oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
            assert_bits_equal(to_np(w), hw[0], f"step {step} master")
            assert_bits_equal(to_np(v), hv[0], f"step {step} momentum")
            for r in (0, P - 1):
                assert_bits_equal(to_np(flat[r]), host[r], f"step {step} grad {r}")
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        red.destroy()
        gar.ar_destroy(comm)


def test_reducer_orders_after_producer_streams():
    """Each gradient is written by a copy on one of three side streams and
    marked ready on that stream, in a shuffled order; the all-reduce must
    see the copied values (an ordering bug would read the zeros)."""
    P = 4
    numels = [1 << 20, 3, 4097, 1 << 21, 768, 1 << 19]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    src = [torch.empty(n, dtype=torch.float32, device=dev()) for _ in range(P)]
    for r, x in enumerate(src):
        wgpu.fill(x, "uniform", 30 + r)
    flat = [torch.zeros(n, dtype=torch.float32, device=dev()) for _ in range(P)]
    grads = [[g[offs[t]:offs[t + 1]] for g in flat] for t in range(len(numels))]
    torch.cuda.synchronize()
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 16 << 20, gar.AR_SUM)
    streams = [torch.cuda.Stream() for _ in range(3)]
    try:
        order = np.random.default_rng(0).permutation(len(numels))
        for k, t in enumerate(order):
            s = streams[k % 3]
            with torch.cuda.stream(s):
                torch.cuda._sleep(2_000_000)        # keep the producer busy for a while
                for r in range(P):
                    grads[t][r].copy_(src[r][offs[t]:offs[t + 1]])
            red.mark_ready(int(t), s)
        main = torch.cuda.current_stream()
        red.finalize(main)
        out = [x.clone() for x in flat]              # on the main stream, after finalize
        torch.cuda.synchronize()
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "uniform", 30), op=oracle.SUM)
    for r in range(P):
        assert_bits_equal(to_np(out[r]), want[r], f"rank {r}")


def test_reducer_finalize_launches_unmarked_buckets():
    P = 2
    numels = [5000, 7000, 9000]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=40)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 4 * 8000, gar.AR_MEAN)
    try:
        assert len(set(red.bucket_of())) == 3
        red.mark_ready(2)        # only the last tensor; the others launch at finalize
        red.finalize()
        torch.cuda.synchronize()
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "normal", 40, std=1e-3), op=oracle.MEAN)
    assert_bits_equal(to_np(flat[1]), want[1], "all buckets")


def test_reducer_learning_rate_schedule_and_errors():
    P = 2
    numels = [1000, 2000]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=50)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 25 << 20, gar.AR_MEAN,
                      sgd=(0.1, 0.9, ws, vs, 0))
    host = host_replicas(P, n, "f32", "normal", 50, std=1e-3)
    hw = [workloads.normal_f32(200, n, std=0.02)]
    hv = [np.zeros(n, np.float32)]
    try:
        for step, lr in enumerate((0.1, 0.05, 0.025)):
            red.set_sgd(lr, 0.9)
            red.mark_ready(1)
            with pytest.raises(gar.GarError) as e:
                red.mark_ready(1)                    # marked twice in one step
            assert e.value.status == gar.AR_ERR_STATE
            red.mark_ready(0)
            red.finalize()
            torch.cuda.synchronize()
            oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(lr, 0.9, hw, hv, 0))
            assert_bits_equal(to_np(w), hw[0], f"step {step}")
        with pytest.raises(gar.GarError) as e:
            red.mark_ready(2)
        assert e.value.status == gar.AR_ERR_INVALID_ARG
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    with pytest.raises(gar.GarError) as e:
        red.handle = 1234
        red.finalize()
    assert e.value.status == gar.AR_ERR_STATE


def test_reducer_mark_ready_many_checks_first():
    P = 2
    numels = [300, 500]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=60)
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 25 << 20, gar.AR_SUM)
    try:
        with pytest.raises(gar.GarError) as e:
            red.mark_ready_many([1, 7])             # 7 is out of range: nothing is marked
        assert e.value.status == gar.AR_ERR_INVALID_ARG
        red.mark_ready_many([1, 0])
        red.finalize()
        torch.cuda.synchronize()
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "normal", 60, std=1e-3), op=oracle.SUM)
    assert_bits_equal(to_np(flat[0]), want[0], "marked together")


def test_reducer_wait_bucket_orders_copy_out():
    """A side stream that waits for bucket b sees that bucket's results; a
    bucket not launched yet is refused."""
    P = 4
    numels = [1 << 20, 1 << 20]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=70)
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 4 << 20, gar.AR_SUM)
    side = torch.cuda.Stream()
    try:
        assert red.bucket_of() == [1, 0]
        with pytest.raises(gar.GarError) as e:
            red.wait_bucket(0, side)
        assert e.value.status == gar.AR_ERR_STATE
        red.mark_ready(1)                     # bucket 0 (the last tensor) launches
        red.wait_bucket(0, side)
        with torch.cuda.stream(side):
            got = flat[2][offs[1]:offs[2]].clone()
        red.finalize()
        torch.cuda.synchronize()
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "normal", 70, std=1e-3), op=oracle.SUM)
    assert_bits_equal(to_np(got), want[2][offs[1]:offs[2]], "copied after wait_bucket")


def test_reducer_step_captured_in_a_cuda_graph():
    """A whole reducer step (marks + finalize) captured into a CUDA graph on
    a capturing stream: the communication streams join the capture through
    the reducer's events; two replays give two oracle steps' bits."""
    P = 8
    numels, offs = _vit_prefix(6_000_000)
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    red = gar.Reducer(comm, grads, numels, gar.AR_BF16, 4 << 20, gar.AR_MEAN,
                      sgd=(0.1, 0.9, ws, vs, 1))
    order = list(range(len(numels) - 1, -1, -1))
    host = host_replicas(P, n, "bf16", "normal", 100, std=1e-3)
    hw = [workloads.normal_f32(200, n, std=0.02)]
    hv = [np.zeros(n, np.float32)]
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):                 # one eager step (warm-up)
            red.mark_ready_many(order, side)
            red.finalize(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            s = torch.cuda.current_stream()
            red.mark_ready_many(order, s)
            red.finalize(s)
        for step in range(2):
            graph.replay()
            torch.cuda.synchronize()
            oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
            assert_bits_equal(to_np(w), hw[0], f"replay {step} master")
            assert_bits_equal(to_np(flat[P - 1]), host[P - 1], f"replay {step} grad")
    finally:
        red.destroy()
        gar.ar_destroy(comm)


def test_reducer_mark_ready_many_refuses_a_repeated_index():
    """A tensor listed twice refuses the whole call and marks nothing."""
    P = 2
    numels = [300, 500]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=61)
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 25 << 20, gar.AR_SUM)
    try:
        with pytest.raises(gar.GarError) as e:
            red.mark_ready_many([1, 0, 1])
        assert e.value.status == gar.AR_ERR_STATE
        red.mark_ready_many([0, 1])                 # nothing was marked: both still free
        red.finalize()
        torch.cuda.synchronize()
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "normal", 61, std=1e-3), op=oracle.SUM)
    assert_bits_equal(to_np(flat[1]), want[1], "after a refused call")


@pytest.mark.parametrize("path", PATHS)
def test_reducer_combined_launches_split_at_table_capacity(path):
    """600 tensors of 1,000 to 1,599 fp32 elements, P = 8, 100 KB buckets
    (24 buckets of about 25 tensors), all marked in one call: the completed
    buckets go out as combined launches, which must split where the table
    holds 256 tensors / 2048 replica pointers.  Two Mean + SGD steps equal
    the oracle's bucket steps, and the last bucket's completion event
    orders a side stream after that bucket's results."""
    P = 8
    rng = np.random.default_rng(62)
    numels = [int(x) for x in rng.integers(1000, 1600, 600)]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=62)
    comm = init(P, gar.AR_MEAN, path)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 100_000, gar.AR_MEAN,
                      sgd=(0.1, 0.9, ws, vs, 1))
    side = torch.cuda.Stream()
    host = host_replicas(P, n, "f32", "normal", 62, std=1e-3)
    hw = workloads.normal_f32(200, n, std=0.02)
    hv = np.zeros(n, np.float32)
    try:
        bucket_of = red.bucket_of()
        nb = len(set(bucket_of))
        assert nb >= 20
        # Expected launches per step: buckets in completion order (0, 1, ...)
        # grouped while a group holds <= 256 tensors and <= 2048 pointers.
        sizes = [bucket_of.count(b) for b in range(nb)]
        groups, segs = 1, 0
        for k in sizes:
            if segs + k > 256 or (segs + k) * P > 2048:
                groups, segs = groups + 1, 0
            segs += k
        assert groups >= 3
        order = list(range(len(numels) - 1, -1, -1))
        for step in range(2):
            before = red.launches()
            red.mark_ready_many(order)
            assert red.launches() - before == groups
            last = bucket_of[0]                     # the bucket of the first tensor completes last
            red.wait_bucket(last, side)
            with torch.cuda.stream(side):
                got_w_side = w.clone()
            red.finalize()
            torch.cuda.synchronize()
            assert gar.ar_get_async_error(comm) == gar.AR_OK
            tens = [[host[r][offs[t]:offs[t + 1]].copy() for r in range(P)] for t in range(len(numels))]
            tw = [hw[offs[t]:offs[t + 1]].copy() for t in range(len(numels))]
            tv = [hv[offs[t]:offs[t + 1]].copy() for t in range(len(numels))]
            for b in range(nb):
                ts = [t for t in range(len(numels)) if bucket_of[t] == b]
                oracle.bucket_all_reduce([tens[t] for t in ts], op=oracle.MEAN,
                                         sgd=(0.1, 0.9, [tw[t] for t in ts], [tv[t] for t in ts], 1))
            hw, hv = np.concatenate(tw), np.concatenate(tv)
            host = [np.concatenate([tens[t][r] for t in range(len(numels))]) for r in range(P)]
            assert_bits_equal(to_np(w), hw, f"step {step} master")
            assert_bits_equal(to_np(v), hv, f"step {step} momentum")
            mine = np.concatenate([np.arange(offs[t], offs[t + 1]) for t in range(len(numels))
                                   if bucket_of[t] == last])
            assert_bits_equal(to_np(got_w_side)[mine], hw[mine],
                              f"step {step} bucket {last} seen after wait_bucket")
            for r in (0, P - 1):
                assert_bits_equal(to_np(flat[r]), host[r], f"step {step} grad {r}")
    finally:
        red.destroy()
        gar.ar_destroy(comm)


def test_reducer_launch_count():
    """Marked one at a time, every bucket launches alone (one launch each);
    marked in one call, the buckets it completes share one launch; the
    counter (ar_reducer_launches) reports exactly that, and both steps give
    the oracle's bits."""
    P = 4
    numels = [40_000] * 12
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, dt="f32", seed=63)
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 4 * 40_000 * 3, gar.AR_SUM)
    try:
        nb = len(set(red.bucket_of()))
        assert nb == 4
        assert red.launches() == 0
        for t in range(len(numels) - 1, -1, -1):
            red.mark_ready(t)
        red.finalize()
        assert red.launches() == nb
        red.mark_ready_many(list(range(len(numels) - 1, -1, -1)))
        red.finalize()
        assert red.launches() == nb + 1
        red.finalize()                              # nothing marked: the buckets launch in finalize
        assert red.launches() == nb + 2
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    host = host_replicas(P, n, "f32", "normal", 63, std=1e-3)
    for _ in range(3):
        host = oracle.all_reduce(host, op=oracle.SUM)
    assert_bits_equal(to_np(flat[2]), host[2], "three Sum steps")


def test_reducer_step_marked_on_one_stream_launches_there():
    """Every tensor marked in one call on a side stream (after a slow
    producer on that stream): the buckets launch on that stream itself.  The
    caller's stream at finalize, and a third stream through wait_bucket,
    still see the results; the next step, marked tensor by tensor on the
    communication-stream path, follows it correctly."""
    P = 4
    numels = [1 << 20, 3, 4097, 1 << 21, 768, 1 << 19]
    offs = np.concatenate([[0], np.cumsum(numels)])
    n = int(offs[-1])
    src = [torch.empty(n, dtype=torch.float32, device=dev()) for _ in range(P)]
    for r, x in enumerate(src):
        wgpu.fill(x, "uniform", 80 + r)
    flat = [torch.zeros(n, dtype=torch.float32, device=dev()) for _ in range(P)]
    grads = [[g[offs[t]:offs[t + 1]] for g in flat] for t in range(len(numels))]
    torch.cuda.synchronize()
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    red = gar.Reducer(comm, grads, numels, gar.AR_F32, 8 << 20, gar.AR_SUM)
    prod, other = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()
    try:
        bucket_of = red.bucket_of()
        assert len(set(bucket_of)) >= 2
        with torch.cuda.stream(prod):
            torch.cuda._sleep(2_000_000)
            for r in range(P):
                flat[r].copy_(src[r])
        red.mark_ready_many(list(range(len(numels) - 1, -1, -1)), prod)
        assert red.launches() == 1
        b0 = bucket_of[0]
        red.wait_bucket(b0, other)
        with torch.cuda.stream(other):
            got = flat[1][offs[0]:offs[1]].clone()
        red.finalize(main)
        out = [x.clone() for x in flat]              # on the main stream, after finalize
        for t in range(len(numels) - 1, -1, -1):     # second step: one bucket per launch
            red.mark_ready(t, main)
        red.finalize(main)
        out2 = [x.clone() for x in flat]
        torch.cuda.synchronize()
        assert red.launches() == 1 + len(set(bucket_of))
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    want = oracle.all_reduce(host_replicas(P, n, "f32", "uniform", 80), op=oracle.SUM)
    assert_bits_equal(to_np(got), want[1][offs[0]:offs[1]], "copied after wait_bucket")
    for r in range(P):
        assert_bits_equal(to_np(out[r]), want[r], f"step 1 rank {r}")
    want2 = oracle.all_reduce([w.copy() for w in want], op=oracle.SUM)
    for r in range(P):
        assert_bits_equal(to_np(out2[r]), want2[r], f"step 2 rank {r}")


def test_reducer_steps_on_one_stream_chain_with_sgd():
    """Four Mean + SGD steps each marked in one call and finalized on the
    same stream, no synchronisation between them (consecutive steps' kernels
    follow each other on that stream): the oracle's bits after four steps."""
    P = 8
    numels, offs = _vit_prefix(3_000_000)
    n = int(offs[-1])
    flat, w, v, grads, ws, vs = _setup(P, numels, offs, seed=150)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    red = gar.Reducer(comm, grads, numels, gar.AR_BF16, 1 << 20, gar.AR_MEAN,
                      sgd=(0.1, 0.9, ws, vs, 1))
    order = list(range(len(numels) - 1, -1, -1))
    s = torch.cuda.Stream()
    try:
        for _ in range(4):
            red.mark_ready_many(order, s)
            red.finalize(s)
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        red.destroy()
        gar.ar_destroy(comm)
    host = host_replicas(P, n, "bf16", "normal", 150, std=1e-3)
    hw = [workloads.normal_f32(200, n, std=0.02)]
    hv = [np.zeros(n, np.float32)]
    for _ in range(4):
        oracle.bucket_all_reduce([host], op=oracle.MEAN, sgd=(0.1, 0.9, hw, hv, 1))
    assert_bits_equal(to_np(w), hw[0], "master")
    assert_bits_equal(to_np(v), hv[0], "momentum")
    for r in (0, 3, P - 1):
        assert_bits_equal(to_np(flat[r]), host[r], f"grad {r}")
