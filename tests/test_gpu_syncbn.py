"""GPU parity of the synchronized batch-norm statistics (ar_syncbn_stats)
against the CPU oracle, bit for bit, and end to end against batch_norm on
the whole batch."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
from gpucase import assert_bits_equal, dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("P", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("C", [1, 64, 2048, 5001])
def test_syncbn_stats_equals_oracle(P, C):
    rng = np.random.default_rng(P * 1000 + C)
    counts = [int(c) for c in rng.integers(1, 5000, size=P)]
    sums = [np.float32(rng.normal(0, 1, C) * c) for c in counts]
    sq = [np.float32(np.abs(rng.normal(1, 0.5, C)) * c + s * s / c) for s, c in zip(sums, counts)]
    d_s = [torch.from_numpy(x).to(dev()) for x in sums]
    d_q = [torch.from_numpy(x).to(dev()) for x in sq]
    d_m = [torch.empty(C, device=dev()) for _ in range(P)]
    d_i = [torch.empty(C, device=dev()) for _ in range(P)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        gar.ar_syncbn_stats(comm, d_s, d_q, counts, d_m, d_i, C, 1e-5)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    want_m, want_i = oracle.syncbn_stats(sums, sq, counts, eps=1e-5)
    for r in range(P):
        assert_bits_equal(to_np(d_m[r]), want_m[r], f"mean {r}")
        nan = np.isnan(want_i[r])
        assert np.array_equal(nan, np.isnan(to_np(d_i[r])))
        assert_bits_equal(to_np(d_i[r])[~nan], want_i[r][~nan], f"invstd {r}")


def test_syncbn_end_to_end_whole_batch():
    """Activations of 4 ranks with uneven shards (N = 3, 5, 2, 6, C = 32,
    8x8); the per-shard sums are taken by torch on the GPU in fp32; the
    pooled statistics equal the oracle's on the same sums bit for bit and
    normalize the whole batch like batch_norm within fp32 round-off."""
    P, C = 4, 32
    g = torch.Generator(device=dev()).manual_seed(0)
    xs = [torch.randn(n, C, 8, 8, device=dev(), generator=g) for n in (3, 5, 2, 6)]
    sums = [x.sum(dim=(0, 2, 3)) for x in xs]
    sq = [(x * x).sum(dim=(0, 2, 3)) for x in xs]
    counts = [x.shape[0] * 64 for x in xs]
    means = [torch.empty(C, device=dev()) for _ in range(P)]
    invs = [torch.empty(C, device=dev()) for _ in range(P)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        gar.ar_syncbn_stats(comm, sums, sq, counts, means, invs, C, 1e-5)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    want_m, want_i = oracle.syncbn_stats([to_np(s) for s in sums], [to_np(q) for q in sq], counts)
    assert_bits_equal(to_np(means[2]), want_m[2], "mean")
    assert_bits_equal(to_np(invs[2]), want_i[2], "invstd")
    whole = torch.cat(xs).double()
    bn = torch.nn.functional.batch_norm(whole, None, None, training=True, eps=1e-5)
    mine = (whole - means[0].double()[None, :, None, None]) * invs[0].double()[None, :, None, None]
    assert float((mine - bn).abs().max()) <= 1e-4


def test_prepared_syncbn_equals_direct_call():
    """ar_syncbn_stats through PreparedCall (pointer and count arrays
    marshalled once, called twice) gives the direct call's bits."""
    P, C = 8, 512
    rng = np.random.default_rng(77)
    counts = [int(c) for c in rng.integers(1, 5000, size=P)]
    sums = [np.float32(rng.normal(0, 1, C) * c) for c in counts]
    sq = [np.float32(np.abs(rng.normal(1, 0.5, C)) * c + s * s / c) for s, c in zip(sums, counts)]
    d_s = [torch.from_numpy(x).to(dev()) for x in sums]
    d_q = [torch.from_numpy(x).to(dev()) for x in sq]
    direct = [[torch.empty(C, device=dev()) for _ in range(P)] for _ in range(2)]
    prepared = [[torch.empty(C, device=dev()) for _ in range(P)] for _ in range(2)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        gar.ar_syncbn_stats(comm, d_s, d_q, counts, direct[0], direct[1], C, 1e-5)
        call = gar.PreparedCall("ar_syncbn_stats", comm, d_s, d_q, counts, prepared[0],
                                prepared[1], C, 1e-5)
        call()
        call()
        torch.cuda.synchronize()
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    for k in range(2):
        for r in range(P):
            assert_bits_equal(to_np(prepared[k][r]), to_np(direct[k][r]), f"output {k} rank {r}")


@pytest.mark.parametrize("P", [2, 3, 8, 16])
def test_syncbn_stats_hard_inputs_equal_oracle(P):
    """Channels chosen to stress the kernel's sums and divisions: ranks'
    sums whose exponents lie close together or far apart, zeros of both
    signs, ranks that cancel exactly, subnormal sums, infinities and NaNs
    (which take the IEEE division), and a pooled count with many significant
    bits; every output against the oracle."""
    C = 4099
    rng = np.random.default_rng(900 + P)
    counts = [int(c) for c in rng.integers(1, 1 << 40, size=P)]
    spread = rng.integers(0, 80, size=C)
    sums, sq = [], []
    for r in range(P):
        mant = rng.uniform(1, 2, size=C) * rng.choice([-1.0, 1.0], size=C)
        expo = rng.integers(-20, 20, size=C) + (rng.integers(0, 1 << 30, size=C) % (spread + 1))
        sums.append(np.float32(np.ldexp(mant, expo)))
        sq.append(np.float32(np.ldexp(rng.uniform(1, 2, size=C), expo + 2)))
    sums, sq = np.stack(sums), np.stack(sq)
    sums[:, 0:40] = 0.0
    sums[:, 0:20] = -0.0
    sums[0, 20:30] = -0.0
    for r in range(1, P, 2):                    # rank r cancels rank r - 1
        sums[r, 40:80] = -sums[r - 1, 40:80]
    sums[:, 80:100] = np.float32(1e-45) * rng.integers(-3, 4, size=(P, 20))
    sums[P - 1, 100] = np.inf
    sums[0, 101] = -np.inf
    sums[P - 1, 102] = np.nan
    sq[0, 103] = np.inf
    sq[P - 1, 104] = np.nan
    sums[0, 105], sums[P - 1, 105] = np.inf, -np.inf
    sums, sq = [np.ascontiguousarray(x) for x in sums], [np.ascontiguousarray(x) for x in sq]
    d_s = [torch.from_numpy(x).to(dev()) for x in sums]
    d_q = [torch.from_numpy(x).to(dev()) for x in sq]
    d_m = [torch.empty(C, device=dev()) for _ in range(P)]
    d_i = [torch.empty(C, device=dev()) for _ in range(P)]
    comm = gar.ar_init(P, 0, gar.AR_SUM)
    try:
        gar.ar_syncbn_stats(comm, d_s, d_q, counts, d_m, d_i, C, 1e-5)
        torch.cuda.synchronize()
    finally:
        gar.ar_destroy(comm)
    want_m, want_i = oracle.syncbn_stats(sums, sq, counts, eps=1e-5)
    for r in range(P):
        for got, want, what in ((to_np(d_m[r]), want_m[r], "mean"), (to_np(d_i[r]), want_i[r], "invstd")):
            nan = np.isnan(want)
            assert np.array_equal(nan, np.isnan(got)), f"{what} {r}: NaN positions"
            assert_bits_equal(got[~nan], want[~nan], f"{what} {r}")
