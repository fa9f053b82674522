"""CPU oracle of the gradient all-reduce -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The product path (``gradient_all_reduce_gb300``) never does,
and the two share no code.

``oracle.c`` is the plain definition of the collectives (all-reduce with Sum
or Mean, reduce-scatter, all-gather, broadcast, the bucketed all-reduce with
its SGD-momentum step, and the bucket assignment); this module compiles it
with gcc and wraps it for NumPy arrays.  ``oracle.mlp`` holds the fp64
4-layer MLP whose per-shard gradients feed the DDP-equivalence check.
Every function cites its source in ``oracle.c``.  Parity is pinned (see the
``-m "not gpu"`` tests): no function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "oracle.c"
LIB = HERE / "liboracle.so"

F32, BF16 = 0, 1
SUM, MEAN = 0, 1
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
LDFLAGS = ["-lm"]


def _stamp(src: Path) -> str:
    return hashlib.sha256(src.read_bytes() + " ".join(CFLAGS).encode()).hexdigest()[:16]


def build(src: Path = SRC, out: Path = LIB) -> Path:
    """Compile ``src`` with gcc into ``out`` unless an up-to-date copy exists."""
    stamp = out.with_suffix(".stamp")
    want = _stamp(src)
    if out.exists() and stamp.exists() and stamp.read_text() == want:
        return out
    tmp = out.with_name(out.name + f".{os.getpid()}.tmp")
    subprocess.run(["gcc", *CFLAGS, "-o", str(tmp), str(src), *LDFLAGS], check=True)
    os.replace(tmp, out)
    stamp.write_text(want)
    return out


_c_ptrs = ctypes.POINTER(ctypes.c_void_p)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
    lib.oracle_f32_to_bf16_array.restype = None
    lib.oracle_all_reduce.argtypes = [ctypes.c_int, _c_ptrs, _c_ptrs, ctypes.c_size_t,
                                      ctypes.c_int, ctypes.c_int]
    lib.oracle_reduce_scatter.argtypes = lib.oracle_all_reduce.argtypes
    lib.oracle_all_gather.argtypes = [ctypes.c_int, _c_ptrs, _c_ptrs, ctypes.c_size_t, ctypes.c_int]
    lib.oracle_broadcast.argtypes = [ctypes.c_int, _c_ptrs, ctypes.c_size_t, ctypes.c_int,
                                     ctypes.c_int]
    lib.oracle_bucket_all_reduce.argtypes = [
        ctypes.c_int, ctypes.c_int, _c_ptrs, ctypes.POINTER(ctypes.c_uint64), ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_float, _c_ptrs, _c_ptrs, ctypes.c_int]
    lib.oracle_bucket_plan.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                                       ctypes.c_uint64, ctypes.POINTER(ctypes.c_int)]
    lib.oracle_bucket_accumulate.argtypes = [
        ctypes.c_int, ctypes.c_int, _c_ptrs, ctypes.POINTER(ctypes.c_uint64), ctypes.c_int,
        _c_ptrs, ctypes.c_float, ctypes.c_int]
    lib.oracle_bucket_all_reduce_accumulated.argtypes = [
        ctypes.c_int, ctypes.c_int, _c_ptrs, ctypes.POINTER(ctypes.c_uint64), ctypes.c_int,
        ctypes.c_int, _c_ptrs, ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_float,
        _c_ptrs, _c_ptrs, ctypes.c_int]
    lib.oracle_syncbn_stats.argtypes = [ctypes.c_int, _c_ptrs, _c_ptrs,
                                        ctypes.POINTER(ctypes.c_uint64), _c_ptrs, _c_ptrs,
                                        ctypes.c_size_t, ctypes.c_float]
    lib.oracle_syncbn_stats.restype = ctypes.c_int
    lib.oracle_sharded_sgd_step.argtypes = [
        ctypes.c_int, _c_ptrs, _c_ptrs, _c_ptrs, _c_ptrs, ctypes.c_size_t, ctypes.c_int,
        ctypes.c_int, ctypes.c_float, ctypes.c_float]
    for f in ("oracle_sharded_sgd_step", "oracle_all_reduce", "oracle_reduce_scatter",
              "oracle_all_gather",
              "oracle_broadcast", "oracle_bucket_all_reduce", "oracle_bucket_plan",
              "oracle_bucket_accumulate", "oracle_bucket_all_reduce_accumulated"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


_LIB: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = _bind(ctypes.CDLL(str(build())))
    return _LIB


def load(path: Path) -> ctypes.CDLL:
    """Load and bind another build of the oracle source (used by the tests
    that check the pins catch planted mistakes)."""
    return _bind(ctypes.CDLL(str(path)))


# ------------------------------------------------------------- wrappers

def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle arrays are float32 or uint16 (bf16 bits), got {a.dtype}")


def _ptrs(arrays) -> ctypes.Array:
    for a in arrays:
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle arrays must be C-contiguous")
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: invalid arguments")


def all_reduce(send, recv=None, op: int = SUM, L=None) -> list[np.ndarray]:
    """All-reduce of the P replicas ``send``; results land in ``recv`` (new
    arrays if None; pass ``recv=send`` for in place)."""
    L = L or lib()
    P, n, dt = len(send), send[0].size, _dtype_code(send[0])
    recv = [np.empty_like(s) for s in send] if recv is None else recv
    _check(L.oracle_all_reduce(P, _ptrs(send), _ptrs(recv), n, dt, op), "all_reduce")
    return recv


def reduce_scatter(send, recv=None, op: int = SUM, L=None) -> list[np.ndarray]:
    L = L or lib()
    P, n, dt = len(send), send[0].size, _dtype_code(send[0])
    if recv is None:
        recv = [np.empty(n // P, dtype=send[0].dtype) for _ in send]
    _check(L.oracle_reduce_scatter(P, _ptrs(send), _ptrs(recv), n, dt, op), "reduce_scatter")
    return recv


def all_gather(send, recv=None, L=None) -> list[np.ndarray]:
    L = L or lib()
    P, shard, dt = len(send), send[0].size, _dtype_code(send[0])
    if recv is None:
        recv = [np.empty(shard * P, dtype=send[0].dtype) for _ in send]
    _check(L.oracle_all_gather(P, _ptrs(send), _ptrs(recv), shard * P, dt), "all_gather")
    return recv


def broadcast(buf, root: int = 0, L=None) -> list[np.ndarray]:
    L = L or lib()
    _check(L.oracle_broadcast(len(buf), _ptrs(buf), buf[0].size, _dtype_code(buf[0]), root),
           "broadcast")
    return buf


def bucket_all_reduce(tensors, op: int = MEAN, sgd=None, L=None) -> None:
    """In-place bucketed all-reduce.  ``tensors[t][r]`` is replica r of
    tensor t.  ``sgd`` = (lr, momentum, master list, momentum list,
    write_back) or None."""
    L = L or lib()
    T = len(tensors)
    if T == 0:
        return
    P = len(tensors[0])
    flat = [a for reps in tensors for a in reps]
    numel = (ctypes.c_uint64 * T)(*[reps[0].size for reps in tensors])
    dt = _dtype_code(flat[0])
    if sgd is None:
        rc = L.oracle_bucket_all_reduce(P, T, _ptrs(flat), numel, dt, op, 0.0, 0.0,
                                        None, None, 1)
    else:
        lr, mom, master, mbuf, wb = sgd
        rc = L.oracle_bucket_all_reduce(P, T, _ptrs(flat), numel, dt, op, lr, mom,
                                        _ptrs(master), _ptrs(mbuf), int(wb))
    _check(rc, "bucket_all_reduce")


def bucket_accumulate(tensors, acc, scale: float, first: bool, L=None) -> None:
    """A micro-batch before the last: acc[t][r] (fp32) = (first ? 0 : acc) +
    fl(scale * tensors[t][r]), in place; no all-reduce."""
    L = L or lib()
    T = len(tensors)
    if T == 0:
        return
    P = len(tensors[0])
    flat = [a for reps in tensors for a in reps]
    accs = [a for reps in acc for a in reps]
    numel = (ctypes.c_uint64 * T)(*[reps[0].size for reps in tensors])
    _check(L.oracle_bucket_accumulate(P, T, _ptrs(flat), numel, _dtype_code(flat[0]),
                                      _ptrs(accs), scale, int(first)), "bucket_accumulate")


def bucket_all_reduce_accumulated(tensors, acc, scale: float, first: bool, op: int = MEAN,
                                  sgd=None, L=None) -> None:
    """The last micro-batch: all-reduce of every rank's acc + fl(scale * g)
    (optionally fused with SGD), results into the gradient replicas."""
    L = L or lib()
    T = len(tensors)
    if T == 0:
        return
    P = len(tensors[0])
    flat = [a for reps in tensors for a in reps]
    accs = [a for reps in acc for a in reps]
    numel = (ctypes.c_uint64 * T)(*[reps[0].size for reps in tensors])
    dt = _dtype_code(flat[0])
    if sgd is None:
        rc = L.oracle_bucket_all_reduce_accumulated(P, T, _ptrs(flat), numel, dt, op, _ptrs(accs),
                                                    scale, int(first), 0.0, 0.0, None, None, 1)
    else:
        lr, mom, master, mbuf, wb = sgd
        rc = L.oracle_bucket_all_reduce_accumulated(P, T, _ptrs(flat), numel, dt, op, _ptrs(accs),
                                                    scale, int(first), lr, mom, _ptrs(master),
                                                    _ptrs(mbuf), int(wb))
    _check(rc, "bucket_all_reduce_accumulated")


def sharded_sgd_step(grads, params, w_shards, v_shards, lr: float, momentum: float,
                     op: int = MEAN, L=None) -> None:
    """ZeRO-1 step: reduce-scatter of grads, each owner's SGD on its fp32
    shard (in place), all-gather of the updated weights into every params
    replica (rounded to the replicas' dtype)."""
    L = L or lib()
    P, n = len(grads), grads[0].size
    _check(L.oracle_sharded_sgd_step(P, _ptrs(grads), _ptrs(params), _ptrs(w_shards),
                                     _ptrs(v_shards), n, _dtype_code(grads[0]), op, lr,
                                     momentum), "sharded_sgd_step")


def syncbn_stats(sums, sqsums, counts, eps: float = 1e-5, L=None):
    """Pooled batch-norm statistics: every rank's (mean, invstd) per channel
    from the ranks' per-channel fp32 sums, sums of squares and counts."""
    L = L or lib()
    P, C = len(sums), sums[0].size
    mean = [np.empty(C, np.float32) for _ in range(P)]
    invstd = [np.empty(C, np.float32) for _ in range(P)]
    cnt = (ctypes.c_uint64 * P)(*[int(c) for c in counts])
    _check(L.oracle_syncbn_stats(P, _ptrs(sums), _ptrs(sqsums), cnt, _ptrs(mean), _ptrs(invstd), C,
                                 eps), "syncbn_stats")
    return mean, invstd


def bucket_plan(nbytes, cap_bytes: int = 25 << 20, L=None) -> list[int]:
    """Bucket index of every tensor (registration order in, reverse fill)."""
    L = L or lib()
    T = len(nbytes)
    out = (ctypes.c_int * max(T, 1))()
    nb = (ctypes.c_uint64 * max(T, 1))(*nbytes)
    k = L.oracle_bucket_plan(T, nb, cap_bytes, out)
    if k < 0:
        raise ValueError("bucket_plan: invalid arguments")
    return list(out)[:T]


def f32_to_bf16(x: np.ndarray, L=None) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns through the oracle."""
    L = L or lib()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(flat.size, dtype=np.uint16)
    L.oracle_f32_to_bf16_array(flat.ctypes.data, out.ctypes.data, flat.size)
    return out.reshape(np.shape(x))
