"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when
the oracle disagrees with: exact integer or rational arithmetic (brute force
with Python integers and fractions), an independent library routine (NumPy
float32 arithmetic, torch's CPU bf16 cast, torch.optim.SGD), values worked
out by hand, or invariants of the collectives.  ``test_oracle_pins`` runs
them on the oracle; ``test_oracle_mutants`` runs them on copies of the
oracle with planted mistakes and requires each copy to fail at least one.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

import oracle
from oracle import MEAN, SUM

SIZES = (0, 1, 2, 3, 5, 8, 17, 33)


def round_to_f32(q: Fraction) -> float:
    """The fp32 nearest to the rational q, ties to even (normal range)."""
    if q == 0:
        return 0.0
    neg, a, e = q < 0, abs(q), 0
    while a >= 2 ** 24:
        a /= 2
        e += 1
    while a < 2 ** 23:
        a *= 2
        e -= 1
    m = math.floor(a)
    rem = a - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    v = math.ldexp(float(m), e)
    return -v if neg else v


def f32(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float32)


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32 if a.dtype == np.float32 else np.uint16)


# ------------------------------------------------------------ all-reduce

def pin_sum_integers_exact(L):
    """Integer-valued inputs whose sums stay below 2**24: every order gives
    the exact integer sum, so the oracle must return it, on every replica."""
    rng = np.random.default_rng(1)
    for P in range(1, 9):
        for n in SIZES:
            xs = [f32(rng.integers(-(1 << 20), 1 << 20, n)) for _ in range(P)]
            out = oracle.all_reduce(xs, op=SUM, L=L)
            want = np.sum([x.astype(np.int64) for x in xs], axis=0) if n else np.zeros(0)
            for r in range(P):
                assert np.array_equal(out[r].astype(np.int64), want), (P, n, r)


def pin_mean_rational_exact(L):
    """Mean of integer-valued inputs is the exact sum (Python ints) divided by
    P and rounded once to fp32: brute force with fractions."""
    rng = np.random.default_rng(2)
    for P in range(1, 9):
        for n in SIZES:
            xs = [f32(rng.integers(-(1 << 20), 1 << 20, n)) for _ in range(P)]
            out = oracle.all_reduce(xs, op=MEAN, L=L)
            for i in range(n):
                s = sum(int(x[i]) for x in xs)
                want = np.float32(round_to_f32(Fraction(s, P)))
                for r in range(P):
                    assert bits(out[r][i:i + 1])[0] == bits(f32([want]))[0], (P, n, i, r)


def pin_rank_order(L):
    """Order-sensitive sums worked out by hand in fp32 (the ulp of 1e8 is 8,
    of 2**24 is 2): only ascending rank order gives these values."""
    cases = [
        ([1e8, 1.0, -1e8, 1.0], 1.0),          # ((1e8+1)=1e8, -1e8 -> 0, +1) = 1
        ([1.0, 1e8, -1e8], 0.0),               # (1+1e8)=1e8, -1e8 -> 0
        ([2.0 ** 24, 1.0, 1.0], 2.0 ** 24),    # each +1 ties back to even 2**24
        ([1.0, 1.0, 2.0 ** 24], 2.0 ** 24 + 2),
        ([3.0, 2.0 ** 24, 2.0 ** 24], 2.0 ** 25 + 4),  # 3+2**24 -> 2**24+4 (tie to even)
    ]
    for vals, want in cases:
        xs = [f32([v]) for v in vals]
        out = oracle.all_reduce(xs, op=SUM, L=L)
        assert float(out[0][0]) == want, (vals, float(out[0][0]), want)


def pin_signed_zero(L):
    """A sum of one term is that term: -0.0 survives when every replica is
    -0.0; +0.0 + -0.0 is +0.0 under round-to-nearest."""
    for P in (1, 2, 3, 8):
        for op in (SUM, MEAN):
            out = oracle.all_reduce([f32([-0.0]) for _ in range(P)], op=op, L=L)
            assert bits(out[0])[0] == 0x80000000, (P, op)
    out = oracle.all_reduce([f32([0.0]), f32([-0.0])], op=SUM, L=L)
    assert bits(out[0])[0] == 0


def numpy_all_reduce(xs, op):
    """Independent route: NumPy float32 elementwise adds in rank order."""
    acc = xs[0].astype(np.float32).copy()
    for x in xs[1:]:
        acc = np.add(acc, x, dtype=np.float32)
    if op == MEAN:
        acc = np.divide(acc, np.float32(len(xs)), dtype=np.float32)
    return acc


def pin_matches_numpy_f32(L):
    """Random fp32 inputs (U(-1,1), N(0,1), mixed magnitudes): bit-exact with
    NumPy's float32 add/divide taken in rank order."""
    rng = np.random.default_rng(3)
    for P in (1, 2, 3, 4, 5, 7, 8, 16):
        n = 4099
        xs = [f32(rng.uniform(-1, 1, n) * 10.0 ** rng.integers(-30, 30, n)) for _ in range(P)]
        for op in (SUM, MEAN):
            out = oracle.all_reduce(xs, op=op, L=L)
            want = numpy_all_reduce(xs, op)
            for r in range(P):
                assert np.array_equal(bits(out[r]), bits(want)), (P, op, r)


def _torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bf16_probe_values() -> np.ndarray:
    """Every upper half (all signs, exponents and kept significands) combined
    with the lower halves that decide rounding: 0, just below, at and above
    one half, odd and even kept parts, all ones; NaNs removed."""
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], np.uint32)
    u = (hi[:, None] | lows[None, :]).ravel()
    f = u.view(np.float32)
    return f[~np.isnan(f)]


def pin_bf16_round_matches_torch(L):
    """fp32 -> bf16 round-to-nearest-even against torch's CPU cast, on the
    probe set (all 2**16 upper halves x the deciding lower halves)."""
    f = bf16_probe_values()
    want = _torch_bf16_bits(f)
    got = oracle.f32_to_bf16(f, L=L)
    assert np.array_equal(got, want), hex(int(f.view(np.uint32)[np.flatnonzero(got != want)[0]]))


def pin_bf16_widen_matches_torch(L):
    """bf16 -> fp32 is exact: compare with torch's CPU widening for every
    non-NaN bf16 pattern."""
    import torch
    h = np.arange(1 << 16, dtype=np.uint16)
    want = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    keep = ~np.isnan(want)
    got = np.array([L.oracle_bf16_to_f32(int(v)) for v in h[keep][::5]], dtype=np.float32)
    assert np.array_equal(bits(got), bits(want[keep][::5]))


def pin_bf16_all_reduce(L):
    """bf16 all-reduce = exact widening, NumPy fp32 rank-order sum (and
    divide), one torch RNE cast at the end; bit-exact."""
    rng = np.random.default_rng(4)
    for P in (1, 2, 3, 4, 8):
        n = 1031
        xs32 = [f32(rng.normal(0, 1, n) * 10.0 ** rng.integers(-3, 3, n)) for _ in range(P)]
        xs = [_torch_bf16_bits(x) for x in xs32]                 # bf16 inputs
        wide = [(x.astype(np.uint32) << 16).view(np.float32) for x in xs]
        for op in (SUM, MEAN):
            out = oracle.all_reduce(xs, op=op, L=L)
            want = _torch_bf16_bits(numpy_all_reduce(wide, op))
            for r in range(P):
                assert np.array_equal(out[r], want), (P, op, r)


# ----------------------------------------------- reduce-scatter / gather

def pin_reduce_scatter_by_hand(L):
    """P=2, N=4: rank 0 keeps elements 0..1 of the sum, rank 1 keeps 2..3."""
    xs = [f32([1, 2, 3, 4]), f32([10, 20, 30, 40])]
    out = oracle.reduce_scatter(xs, op=SUM, L=L)
    assert out[0].tolist() == [11, 22] and out[1].tolist() == [33, 44]
    out = oracle.reduce_scatter(xs, op=MEAN, L=L)
    assert out[0].tolist() == [5.5, 11] and out[1].tolist() == [16.5, 22]


def pin_all_gather_by_hand(L):
    """P=3: every rank receives shard 0 ++ shard 1 ++ shard 2."""
    xs = [f32([1, 2]), f32([3, 4]), f32([5, 6])]
    out = oracle.all_gather(xs, L=L)
    for r in range(3):
        assert out[r].tolist() == [1, 2, 3, 4, 5, 6], r


def pin_rs_then_ag_is_all_reduce(L):
    """Invariant: all-gather(reduce-scatter(x)) == all-reduce(x), bit for bit
    (the two halves of the ring all-reduce)."""
    rng = np.random.default_rng(5)
    for P in (1, 2, 4, 8):
        for dt in ("f32", "bf16"):
            n = 24 * P
            xs = [f32(rng.normal(0, 1, n)) for _ in range(P)]
            if dt == "bf16":
                xs = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in xs]
            for op in (SUM, MEAN):
                ar = oracle.all_reduce(xs, op=op, L=L)
                ag = oracle.all_gather(oracle.reduce_scatter(xs, op=op, L=L), L=L)
                for r in range(P):
                    assert np.array_equal(ag[r], ar[r]), (P, dt, op, r)


def pin_broadcast(L):
    """After a broadcast every replica holds the root's bytes; the root is
    unchanged."""
    rng = np.random.default_rng(6)
    for P in (1, 2, 5):
        for root in range(P):
            xs = [f32(rng.normal(0, 1, 9)) for _ in range(P)]
            ref = xs[root].copy()
            oracle.broadcast(xs, root=root, L=L)
            for r in range(P):
                assert np.array_equal(bits(xs[r]), bits(ref)), (P, root, r)


def pin_in_place_all_reduce(L):
    """In place (recv = send) gives the same bits as out of place."""
    rng = np.random.default_rng(7)
    xs = [f32(rng.normal(0, 1, 37)) for _ in range(4)]
    want = oracle.all_reduce(xs, op=MEAN, L=L)
    ys = [x.copy() for x in xs]
    oracle.all_reduce(ys, recv=ys, op=MEAN, L=L)
    for r in range(4):
        assert np.array_equal(bits(ys[r]), bits(want[r]))


# ---------------------------------------------------------- buckets, SGD

def pin_bucket_equals_per_tensor(L):
    """A bucket of several tensors reduces each exactly as its own
    all-reduce would (the operation is elementwise)."""
    rng = np.random.default_rng(8)
    P, sizes = 4, (1, 7, 64, 1000, 3)
    tensors = [[f32(rng.normal(0, 1, n)) for _ in range(P)] for n in sizes]
    want = [oracle.all_reduce(reps, op=MEAN, L=L) for reps in tensors]
    oracle.bucket_all_reduce(tensors, op=MEAN, L=L)
    for t, reps in enumerate(tensors):
        for r in range(P):
            assert np.array_equal(bits(reps[r]), bits(want[t][r])), (t, r)


def pin_sgd_closed_form(L):
    """One replica (P=1) with gradient 1 and v = 0: the first step gives
    v = 1 and w = w - fl(0.1f); the second v = fl(fl(0.9f * 1) + 1) and
    w = w - fl(0.1f * v), worked out with NumPy float32 scalars."""
    lr, mu = np.float32(0.1), np.float32(0.9)
    g = [[f32([1.0, 1.0])]]
    w, v = [f32([0.5, -2.0])], [f32([0.0, 0.0])]
    w0 = w[0].copy()
    oracle.bucket_all_reduce(g, op=SUM, sgd=(lr, mu, w, v, 0), L=L)
    assert v[0].tolist() == [1.0, 1.0]
    assert np.array_equal(w[0], w0 - lr)
    v1 = np.float32(np.float32(mu * np.float32(1.0)) + np.float32(1.0))
    w1 = w[0].copy()
    oracle.bucket_all_reduce([[f32([1.0, 1.0])]], op=SUM, sgd=(lr, mu, w, v, 0), L=L)
    assert np.array_equal(v[0], f32([v1, v1]))
    assert np.array_equal(w[0], w1 - np.float32(lr * v1))


def pin_sgd_matches_torch(L):
    """Momentum SGD against torch.optim.SGD(lr=0.1, momentum=0.9) on CPU, fed
    the same reduced gradient, one step at a time from a common state (torch
    is reset to the oracle's w and v before each step, so differences do not
    compound).  v must agree bit for bit (torch computes fl(fl(0.9 v) + g)
    too); w within 2 ulp of max(|w|, |lr v|), since torch may fuse
    w - lr*v into one rounding."""
    import torch
    rng = np.random.default_rng(9)
    P, n = 4, 513
    w = [f32(rng.normal(0, 0.02, n))]
    v = [np.zeros(n, np.float32)]
    for step in range(3):
        reps = [f32(rng.normal(0, 1e-3, n)) for _ in range(P)]
        g = numpy_all_reduce(reps, MEAN)
        p = torch.nn.Parameter(torch.from_numpy(w[0].copy()))
        opt = torch.optim.SGD([p], lr=0.1, momentum=0.9, foreach=False)
        if step > 0:
            opt.state[p]["momentum_buffer"] = torch.from_numpy(v[0].copy())
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        w_old = w[0].copy()
        oracle.bucket_all_reduce([reps], op=MEAN, sgd=(0.1, 0.9, w, v, 1), L=L)
        assert np.array_equal(bits(reps[0]), bits(g)), step      # write-back = reduced g
        assert np.array_equal(bits(v[0]), bits(opt.state[p]["momentum_buffer"].numpy())), step
        scale = np.maximum(np.abs(w_old), np.abs(np.float32(0.1) * v[0]))
        err = np.abs(w[0].astype(np.float64) - p.detach().numpy().astype(np.float64))
        assert np.all(err <= 2 * np.spacing(scale).astype(np.float64)), step


def pin_sgd_write_back_flag(L):
    """write_back=0 leaves the gradient replicas untouched; 1 overwrites them
    with the reduced gradient."""
    reps = [f32([1.0, 2.0]), f32([3.0, 4.0])]
    w, v = [f32([0, 0])], [f32([0, 0])]
    oracle.bucket_all_reduce([reps], op=MEAN, sgd=(0.1, 0.9, w, v, 0), L=L)
    assert reps[0].tolist() == [1, 2] and reps[1].tolist() == [3, 4]
    oracle.bucket_all_reduce([reps], op=MEAN, sgd=(0.1, 0.9, w, v, 1), L=L)
    assert reps[0].tolist() == [2, 3] and reps[1].tolist() == [2, 3]


def pin_bucket_plan(L):
    """Hand cases of the reverse-order greedy fill with a cap of 10 bytes,
    plus the rule's invariants on the ViT-B/16 gradient set."""
    assert oracle.bucket_plan([4, 4, 4], 10, L=L) == [1, 0, 0]        # fill from the end
    assert oracle.bucket_plan([3, 12, 3], 10, L=L) == [2, 1, 0]       # oversized: alone
    assert oracle.bucket_plan([5, 5, 5, 5], 10, L=L) == [1, 1, 0, 0]  # exactly the cap fits
    assert oracle.bucket_plan([], 10, L=L) == []
    import workloads
    nb = [2 * n for n in workloads.vit_b16_numels()]
    cap = 25 << 20
    plan = oracle.bucket_plan(nb, cap, L=L)
    k = max(plan) + 1
    assert plan[-1] == 0 and all(plan[t] >= plan[t + 1] for t in range(len(plan) - 1))
    fill = [0] * k
    for t, b in enumerate(plan):
        fill[b] += nb[t]
    for b in range(k):
        members = [t for t in range(len(plan)) if plan[t] == b]
        assert fill[b] <= cap or len(members) == 1
        if b + 1 < k:  # greedy: the next tensor would not have fitted
            nxt = max(t for t in range(len(plan)) if plan[t] == b + 1)
            assert fill[b] + nb[nxt] > cap


# ------------------------------------------------- accumulation (no_sync)

def _accumulate_then_reduce(grads, scale, op, L, sgd=None):
    """grads[m][t][r]: micro-batch m's gradient.  Accumulate every
    micro-batch but the last, all-reduce on the last.  Returns (the reduced
    gradient replicas of the last micro-batch, the accumulators)."""
    M = len(grads)
    # stale values from an earlier cycle: the first micro-batch must overwrite them
    acc = [[np.full(x.size, 7.0, np.float32) for x in reps] for reps in grads[0]]
    for m in range(M - 1):
        oracle.bucket_accumulate(grads[m], acc, scale, m == 0, L=L)
    last = [[x.copy() for x in reps] for reps in grads[M - 1]]
    oracle.bucket_all_reduce_accumulated(last, acc, scale, M == 1, op=op, sgd=sgd, L=L)
    return last, acc


def pin_accumulation_undivided_is_m_times(L):
    """The page's check: accumulating M micro-batch gradients without
    dividing by M gives exactly M times the gradient.  Integer-valued
    gradients keep every sum exact, so the results equal the exact integer
    sums (brute force) and differ by exactly the factor M = 4."""
    rng = np.random.default_rng(10)
    P, M, sizes = 3, 4, (5, 17)
    grads = [[[f32(rng.integers(-1000, 1000, n)) for _ in range(P)] for n in sizes]
             for _ in range(M)]
    undivided, _ = _accumulate_then_reduce(grads, 1.0, SUM, L)
    divided, _ = _accumulate_then_reduce(grads, 1.0 / M, SUM, L)
    for t, n in enumerate(sizes):
        exact = np.sum([[g[t][r].astype(np.int64) for r in range(P)] for g in grads], axis=(0, 1))
        for r in range(P):
            assert np.array_equal(undivided[t][r].astype(np.int64), exact), (t, r)
            assert np.array_equal(undivided[t][r], np.float32(M) * divided[t][r]), (t, r)


def pin_accumulation_matches_numpy(L):
    """Random gradients, scale 1/3: the accumulators and the reduced result
    equal NumPy float32 arithmetic taken in the same order, bit for bit."""
    rng = np.random.default_rng(11)
    P, M, n = 4, 3, 1001
    scale = np.float32(1.0 / 3.0)
    for dt in ("f32", "bf16"):
        g32 = [[[f32(rng.normal(0, 1, n))] for _ in range(P)] for _ in range(M)]
        grads = [[[x[0] if dt == "f32" else (x[0].view(np.uint32) >> 16).astype(np.uint16)
                   for x in reps]] for reps in g32]
        wide = [[(x if x.dtype == np.float32 else (x.astype(np.uint32) << 16).view(np.float32))
                 for x in reps[0]] for reps in grads]
        for op in (SUM, MEAN):
            out, acc = _accumulate_then_reduce(grads, float(scale), op, L)
            want_acc = [np.multiply(scale, wide[0][r], dtype=np.float32) for r in range(P)]
            for m in range(1, M - 1):
                want_acc = [np.add(want_acc[r], np.multiply(scale, wide[m][r], dtype=np.float32),
                                   dtype=np.float32) for r in range(P)]
            totals = [np.add(want_acc[r], np.multiply(scale, wide[M - 1][r], dtype=np.float32),
                             dtype=np.float32) for r in range(P)]
            y = numpy_all_reduce(totals, op)
            want = y if dt == "f32" else _torch_bf16_bits(y)
            for r in range(P):
                assert np.array_equal(bits(acc[0][r]), bits(want_acc[r])), (dt, op, r)
                assert np.array_equal(bits(out[0][r]), bits(want)), (dt, op, r)


def pin_accumulation_single_micro_batch_is_all_reduce(L):
    """M = 1 with scale 1 is the plain all-reduce (and leaves acc alone)."""
    rng = np.random.default_rng(12)
    P = 5
    xs = [f32(rng.normal(0, 1, 77)) for _ in range(P)]
    want = oracle.all_reduce(xs, op=MEAN, L=L)
    acc = [[np.full(77, 7.0, np.float32) for _ in range(P)]]
    last = [[x.copy() for x in xs]]
    oracle.bucket_all_reduce_accumulated(last, acc, 1.0, True, op=MEAN, L=L)
    for r in range(P):
        assert np.array_equal(bits(last[0][r]), bits(want[r])), r
        assert np.all(acc[0][r] == 7.0)


def pin_accumulation_with_sgd(L):
    """The fused SGD step on the accumulated gradient equals the SGD step of
    the bucketed all-reduce fed the per-rank totals (acc + scale g), over
    two optimizer steps (so the momentum term matters)."""
    rng = np.random.default_rng(13)
    P, M, n = 2, 2, 300
    w0 = f32(rng.normal(0, 0.02, n))
    for wb in (0, 1):
        w, v = [w0.copy()], [np.zeros(n, np.float32)]
        w2, v2 = [w0.copy()], [np.zeros(n, np.float32)]
        for step in range(2):
            grads = [[[f32(rng.normal(0, 1e-3, n)) for _ in range(P)]] for _ in range(M)]
            out, _ = _accumulate_then_reduce(grads, 0.5, MEAN, L, sgd=(0.1, 0.9, w, v, wb))
            totals = [np.add(np.multiply(np.float32(0.5), grads[0][0][r], dtype=np.float32),
                             np.multiply(np.float32(0.5), grads[1][0][r], dtype=np.float32),
                             dtype=np.float32) for r in range(P)]
            ref = [[x.copy() for x in totals]]
            oracle.bucket_all_reduce(ref, op=MEAN, sgd=(0.1, 0.9, w2, v2, wb), L=L)
            assert np.array_equal(bits(w[0]), bits(w2[0])), (wb, step)
            assert np.array_equal(bits(v[0]), bits(v2[0])), (wb, step)
            want = ref[0][0] if wb else grads[1][0][0]
            assert np.array_equal(bits(out[0][0]), bits(want)), (wb, step)


# ------------------------------------------------------- ZeRO-1 step

def pin_sharded_step_equals_replicated_step(L):
    """Sharding the optimizer state changes no number: the shards of w and v
    after the sharded step, laid end to end, equal w and v after the
    replicated step (every rank updating all of w), and every rank's params
    equal the rounded w (torch's cast for bf16)."""
    rng = np.random.default_rng(14)
    for P in (1, 2, 4, 8):
        for dt in ("f32", "bf16"):
            n = 24 * P
            s = n // P
            g32 = [f32(rng.normal(0, 1e-3, n)) for _ in range(P)]
            grads = g32 if dt == "f32" else [(x.view(np.uint32) >> 16).astype(np.uint16)
                                              for x in g32]
            w0 = f32(rng.normal(0, 0.02, n))
            v0 = f32(rng.normal(0, 1e-3, n))
            ws = [w0[r * s:(r + 1) * s].copy() for r in range(P)]
            vs = [v0[r * s:(r + 1) * s].copy() for r in range(P)]
            params = [np.zeros(n, grads[0].dtype) for _ in range(P)]
            oracle.sharded_sgd_step(grads, params, ws, vs, 0.1, 0.9, op=MEAN, L=L)
            wf, vf = [w0.copy()], [v0.copy()]
            oracle.bucket_all_reduce([[x.copy() for x in grads]], op=MEAN,
                                     sgd=(0.1, 0.9, wf, vf, 0), L=L)
            assert np.array_equal(bits(np.concatenate(ws)), bits(wf[0])), (P, dt)
            assert np.array_equal(bits(np.concatenate(vs)), bits(vf[0])), (P, dt)
            want = wf[0] if dt == "f32" else _torch_bf16_bits(wf[0])
            for q in range(P):
                assert np.array_equal(bits(params[q]), bits(want)), (P, dt, q)


def pin_sharded_step_is_rs_sgd_ag(L):
    """For fp32 gradients the step is its three collectives in a row:
    reduce-scatter, the owner's SGD on its shard (NumPy float32, separate
    roundings), all-gather of the updated shards."""
    rng = np.random.default_rng(15)
    P, n = 4, 64
    s = n // P
    grads = [f32(rng.normal(0, 1, n)) for _ in range(P)]
    w0 = [f32(rng.normal(0, 0.02, s)) for _ in range(P)]
    ws = [x.copy() for x in w0]
    vs = [np.zeros(s, np.float32) for _ in range(P)]
    params = [np.zeros(n, np.float32) for _ in range(P)]
    oracle.sharded_sgd_step(grads, params, ws, vs, 0.1, 0.9, op=SUM, L=L)
    shards = oracle.reduce_scatter(grads, op=SUM, L=L)
    new = []
    for r in range(P):
        v = np.add(np.multiply(np.float32(0.9), np.zeros(s, np.float32)), shards[r],
                   dtype=np.float32)
        new.append(np.subtract(w0[r], np.multiply(np.float32(0.1), v), dtype=np.float32))
        assert np.array_equal(bits(vs[r]), bits(v)), r
    gathered = oracle.all_gather(new, L=L)
    for q in range(P):
        assert np.array_equal(bits(params[q]), bits(gathered[q])), q


# ------------------------------------------------- SyncBN statistics

def _shard_stats(xs):
    """Per-channel fp32 sums of x and x*x and the count, for shards of shape
    (N_r, C, H, W) holding integer values (exact in fp32)."""
    sums = [f32(x.sum(axis=(0, 2, 3))) for x in xs]
    sq = [f32((x * x).sum(axis=(0, 2, 3))) for x in xs]
    counts = [x.shape[0] * x.shape[2] * x.shape[3] for x in xs]
    return sums, sq, counts


def pin_syncbn_equals_whole_batch(L):
    """The page's check: statistics pooled from the shards' sums equal batch
    normalization's statistics on the whole batch (torch's own batch_norm in
    fp64, training mode, biased variance) -- here to within one fp32 rounding
    of the exact values, with uneven shards."""
    import torch
    rng = np.random.default_rng(16)
    C = 8
    xs = [rng.integers(-20, 20, (n, C, 3, 2)).astype(np.float64) for n in (3, 5, 1, 7)]
    sums, sq, counts = _shard_stats(xs)
    mean, invstd = oracle.syncbn_stats(sums, sq, counts, eps=1e-5, L=L)
    whole = torch.from_numpy(np.concatenate(xs))
    m = whole.mean(dim=(0, 2, 3)).numpy()
    v = whole.var(dim=(0, 2, 3), unbiased=False).numpy()
    want_is = 1.0 / np.sqrt(v + np.float64(np.float32(1e-5)))
    for r in range(len(xs)):
        assert np.all(np.abs(mean[r].astype(np.float64) - m) <= np.spacing(np.abs(f32(m)))), r
        assert np.all(np.abs(invstd[r].astype(np.float64) - want_is)
                      <= np.spacing(f32(want_is))), r
    # normalizing the whole batch with the pooled statistics matches batch_norm
    bn = torch.nn.functional.batch_norm(whole, None, None, training=True,
                                        eps=float(np.float32(1e-5))).numpy()
    mine = (np.concatenate(xs) - mean[0].astype(np.float64)[None, :, None, None]) * \
        invstd[0].astype(np.float64)[None, :, None, None]
    assert np.max(np.abs(mine - bn)) <= 1e-5


def pin_syncbn_exact_sums(L):
    """Hand case: two ranks, one channel, values {1, 3} and {5, 7}: n = 4,
    mean = 4, var = (1 + 9 + 25 + 49) / 4 - 16 = 5, invstd = 1/sqrt(5 + eps)."""
    sums = [f32([4.0]), f32([12.0])]
    sq = [f32([10.0]), f32([74.0])]
    mean, invstd = oracle.syncbn_stats(sums, sq, [2, 2], eps=0.0, L=L)
    assert mean[0][0] == 4.0 and mean[1][0] == 4.0
    assert invstd[1][0] == np.float32(1.0 / np.sqrt(5.0))


ALL_PINS = [
    pin_sum_integers_exact, pin_mean_rational_exact, pin_rank_order, pin_signed_zero,
    pin_matches_numpy_f32, pin_bf16_round_matches_torch, pin_bf16_widen_matches_torch,
    pin_bf16_all_reduce, pin_reduce_scatter_by_hand, pin_all_gather_by_hand,
    pin_rs_then_ag_is_all_reduce, pin_broadcast, pin_in_place_all_reduce,
    pin_bucket_equals_per_tensor, pin_sgd_closed_form, pin_sgd_matches_torch,
    pin_sgd_write_back_flag, pin_bucket_plan, pin_accumulation_undivided_is_m_times,
    pin_accumulation_matches_numpy, pin_accumulation_single_micro_batch_is_all_reduce,
    pin_accumulation_with_sgd, pin_sharded_step_equals_replicated_step,
    pin_sharded_step_is_rs_sgd_ag, pin_syncbn_equals_whole_batch, pin_syncbn_exact_sums,
]
