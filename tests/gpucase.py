"""Helpers of the GPU parity tests: replicas made on the device by the
seeded generator, the same inputs regenerated on the host for the oracle,
and bitwise comparison."""
from __future__ import annotations

import os

import numpy as np
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from workloads import gpu as wgpu

DT = {"f32": gar.AR_F32, "bf16": gar.AR_BF16}
OP = {"sum": gar.AR_SUM, "mean": gar.AR_MEAN}
ORACLE_OP = {"sum": oracle.SUM, "mean": oracle.MEAN}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


PATHS = ("ldg", "tma")   # register-staged k_reduce, bulk-copy pipelined k_reduce_tma


def init(P: int, op: int = gar.AR_MEAN, path: str | None = None) -> int:
    """ar_init with the reduce and copy kernels forced to ``path`` (read at
    init): "ldg" for the register-staged kernels, "tma" for the bulk-copy
    pipelines."""
    keys = ("GAR_KERNEL", "GAR_COPY")
    old = {k: os.environ.get(k) for k in keys}
    if path is not None:
        for k in keys:
            os.environ[k] = path
    try:
        return gar.ar_init(P, 0, op)
    finally:
        for k in keys:
            if old[k] is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = old[k]


def dev():
    return torch.device("cuda:0")


def empty(n: int, dt: str, offset: int = 0) -> torch.Tensor:
    """A device buffer of n elements starting ``offset`` elements into its
    allocation (offset 1 gives a pointer that is not 16-byte aligned)."""
    base = torch.empty(n + offset, dtype=TORCH_DT[dt], device=dev())
    return base[offset:]


def replicas(P: int, n: int, dt: str, kind: str = "uniform", seed0: int = 0, std: float = 1.0,
             offset: int = 0) -> list[torch.Tensor]:
    """Replica r: draws of stream seed0 + r, made on the device."""
    out = []
    for r in range(P):
        t = empty(n, dt, offset)
        wgpu.fill(t, kind, seed0 + r, std=std)
        out.append(t)
    return out


def host_replicas(P: int, n: int, dt: str, kind: str = "uniform", seed0: int = 0,
                  std: float = 1.0, idx: np.ndarray | None = None) -> list[np.ndarray]:
    """The same inputs on the host (all n elements, or the elements at idx)."""
    return [workloads.replica_values(kind, dt, seed0 + r, n, std=std, idx=idx) for r in range(P)]


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    g, w = bits(got), bits(want)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{what}: {bad.size} of {g.size} elements differ; first at {bad[0]}: "
                             f"got {g[bad[0]]:#x}, want {w[bad[0]]:#x}")


def gather(t: torch.Tensor, idx: np.ndarray) -> np.ndarray:
    """Elements of device tensor t at host indices idx."""
    it = torch.from_numpy(idx.astype(np.int64)).to(t.device)
    return to_np(t[it])


def sample_indices(n: int, k: int, seed: int, extra=()) -> np.ndarray:
    """k random positions plus both ends and any given positions, sorted."""
    rng = np.random.default_rng(seed)
    pos = set(int(i) for i in rng.integers(0, n, size=min(k, n)))
    pos.update(i for i in (0, n - 1, *extra) if 0 <= i < n)
    return np.array(sorted(pos), dtype=np.uint64)


def bits_equal_device(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality of two device tensors of the same dtype."""
    view = torch.int32 if a.dtype == torch.float32 else torch.int16
    return bool(torch.equal(a.view(view), b.view(view)))
