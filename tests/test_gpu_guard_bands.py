"""Guard bands: every buffer a call is given sits inside a larger allocation
whose bytes before and after it hold a canary pattern, and after the call
the canaries must be intact.  This stands in for a device-side bounds
checker on the write side: a kernel that stores one byte outside the ranges
it was given fails here.  Every entry point, both kernel paths (the
register-staged kernels and the bulk-copy pipelines), ragged and tiny sizes,
and buffers that start off a 16-byte boundary."""
import pytest
import torch

import gradient_all_reduce_gb300 as gar
from gpucase import DT, PATHS, TORCH_DT, dev, init
from workloads import gpu as wgpu

pytestmark = pytest.mark.gpu

GUARD = 256          # bytes of canary on each side (two 128-byte lines)
CANARY = 0xA5
SIZES = [1, 3, 17, 4097, 70_001]


class Guarded:
    """n elements of dtype dt inside canary bands; ``offset`` extra elements
    before the buffer make its start unaligned."""

    def __init__(self, n: int, dt: str, offset: int = 0):
        self.es = 4 if dt == "f32" else 2
        self.pad = GUARD // self.es + offset
        self.base = torch.empty(self.pad + n + GUARD // self.es, dtype=TORCH_DT[dt], device=dev())
        self.base.view(torch.uint8).fill_(CANARY)
        self.t = self.base[self.pad:self.pad + n]
        self.n = n

    def intact(self) -> bool:
        b = self.base.view(torch.uint8)
        lo, hi = self.pad * self.es, (self.pad + self.n) * self.es
        return bool((b[:lo] == CANARY).all()) and bool((b[hi:] == CANARY).all())


def filled(n, dt, seed, offset=0, kind="uniform", std=1.0):
    g = Guarded(n, dt, offset)
    wgpu.fill(g.t, kind, seed, std=std)
    return g


def zeros(n, dt="f32", offset=0):
    g = Guarded(n, dt, offset)
    g.t.zero_()
    return g


def check(bufs, what):
    torch.cuda.synchronize()
    bad = [i for i, b in enumerate(bufs) if not b.intact()]
    assert not bad, f"{what}: canary overwritten around buffers {bad}"


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("P", [3, 8])
def test_collectives_write_only_their_buffers(path, dt, P):
    comm = init(P, gar.AR_MEAN, path)
    try:
        for n in SIZES:
            for off in (0, 1):
                xs = [filled(n, dt, r, off) for r in range(P)]
                gar.ar_all_reduce(comm, [x.t for x in xs], [x.t for x in xs], n, DT[dt], gar.AR_MEAN)
                check(xs, f"AR in place n={n} off={off}")
                ys = [Guarded(n, dt, off) for _ in range(P)]
                gar.ar_all_reduce(comm, [x.t for x in xs], [y.t for y in ys], n, DT[dt], gar.AR_SUM)
                check(xs + ys, f"AR out of place n={n} off={off}")
                gar.ar_broadcast(comm, [x.t for x in xs], n, DT[dt], P - 1)
                check(xs, f"BC n={n} off={off}")
                m = n  # shard length: the full count is P * n
                full = [filled(P * m, dt, 10 + r, off) for r in range(P)]
                shards = [Guarded(m, dt, off) for _ in range(P)]
                gar.ar_reduce_scatter(comm, [f.t for f in full], [s.t for s in shards], P * m, DT[dt],
                                      gar.AR_MEAN)
                check(full + shards, f"RS n={P * m} off={off}")
                out = [Guarded(P * m, dt, off) for _ in range(P)]
                gar.ar_all_gather(comm, [s.t for s in shards], [o.t for o in out], P * m, DT[dt])
                check(shards + out, f"AG n={P * m} off={off}")
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("P", [3, 8])
def test_bucket_sgd_and_accumulation_write_only_their_buffers(path, dt, P):
    comm = init(P, gar.AR_MEAN, path)
    try:
        for off in (0, 1):
            grads = [[filled(n, dt, 100 * t + r, off, "normal", 1e-3) for r in range(P)]
                     for t, n in enumerate(SIZES)]
            ws = [filled(n, "f32", 200 + t, off, "normal", 0.02) for t, n in enumerate(SIZES)]
            vs = [zeros(n, "f32", off) for n in SIZES]
            accs = [[zeros(n, "f32", off) for _ in range(P)] for n in SIZES]
            every = [g for reps in grads for g in reps] + ws + vs + [a for reps in accs for a in reps]
            g_t = [[g.t for g in reps] for reps in grads]
            a_t = [[a.t for a in reps] for reps in accs]
            sgd = (0.1, 0.9, [w.t for w in ws], [v.t for v in vs], 1)
            gar.ar_bucket_all_reduce(comm, g_t, SIZES, DT[dt], gar.AR_MEAN, sgd=sgd)
            check(every, f"bucket + SGD off={off}")
            gar.ar_bucket_accumulate(comm, g_t, SIZES, DT[dt], a_t, 0.5, True)
            check(every, f"first micro-batch off={off}")
            gar.ar_bucket_accumulate(comm, g_t, SIZES, DT[dt], a_t, 0.5, False)
            check(every, f"later micro-batch off={off}")
            gar.ar_bucket_all_reduce_accumulated(comm, g_t, SIZES, DT[dt], a_t, 0.5, False,
                                                 gar.AR_MEAN, sgd=sgd)
            check(every, f"last micro-batch + SGD off={off}")
            gar.ar_bucket_all_reduce_accumulated(comm, g_t, SIZES, DT[dt], a_t, 0.5, False,
                                                 gar.AR_SUM)
            check(every, f"last micro-batch off={off}")
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("P", [3, 8])
def test_sharded_step_writes_only_its_buffers(path, dt, P):
    comm = init(P, gar.AR_MEAN, path)
    try:
        for m in SIZES:
            for off in (0, 1):
                n = P * m
                grads = [filled(n, dt, r, off, "normal", 1e-3) for r in range(P)]
                params = [Guarded(n, dt, off) for _ in range(P)]
                ws = [filled(m, "f32", 300 + r, off, "normal", 0.02) for r in range(P)]
                vs = [zeros(m, "f32", off) for _ in range(P)]
                gar.ar_sharded_sgd_step(comm, [g.t for g in grads], [p.t for p in params],
                                        [w.t for w in ws], [v.t for v in vs], n, DT[dt], 0.1, 0.9,
                                        gar.AR_MEAN)
                check(grads + params + ws + vs, f"ZeRO-1 step n={n} off={off}")
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)


@pytest.mark.parametrize("P", [1, 3, 8, 16])
def test_syncbn_and_noalloc_write_only_their_buffers(P):
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        for C in (1, 3, 64, 2049):
            sums = [filled(C, "f32", r) for r in range(P)]
            sq = [filled(C, "f32", 50 + r) for r in range(P)]
            for s in sq:
                s.t.abs_().add_(1.0)
            means = [Guarded(C, "f32") for _ in range(P)]
            inv = [Guarded(C, "f32") for _ in range(P)]
            gar.ar_syncbn_stats(comm, [s.t for s in sums], [s.t for s in sq], [1000] * P,
                                [m.t for m in means], [i.t for i in inv], C, 1e-5)
            check(sums + sq + means + inv, f"SyncBN C={C}")
        assert gar.ar_get_async_error(comm) == gar.AR_OK
    finally:
        gar.ar_destroy(comm)
    for n in SIZES:
        xs = [filled(n, "f32", r) for r in range(P)]
        gar.ar_all_reduce_noalloc(P, [x.t for x in xs], [x.t for x in xs], n, gar.AR_F32,
                                  gar.AR_MEAN)
        check(xs, f"no-alloc AR n={n}")


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_the_canary_check_sees_one_stray_byte(dt):
    """The detector itself: one byte changed just before or just after the
    buffer (by torch, not by a kernel under test) is caught; a write inside
    the buffer is not."""
    for where in ("before", "after", "inside"):
        g = Guarded(17, dt, 1)
        lo, hi = g.pad * g.es, (g.pad + g.n) * g.es
        pos = {"before": lo - 1, "after": hi, "inside": hi - 1}[where]
        g.base.view(torch.uint8)[pos] = 0
        assert g.intact() == (where == "inside"), where
