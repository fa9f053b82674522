"""Python binding of libgar.so, the GB300 gradient all-reduce library.

Argument marshalling only: every function forwards to the C entry point of
the same name declared in ``include/gar.h``; all work runs in the library's
CUDA kernels.  Buffers may be given as raw device addresses (int) or as
objects with ``data_ptr()`` (torch tensors); streams as raw handles (int),
objects with ``cuda_stream`` (torch.cuda.Stream), or None for the current
torch stream (the legacy default stream when torch is not imported).

The library must be built first (``gradient_all_reduce_gb300.build.build()``
or ``__graft_entry__.build()``).  It is loaded on first use; without it
every call raises ImportError -- there is no fallback implementation.
``GAR_LIBRARY=debug`` in the environment loads the debug build instead
(``build(debug=True)``: the same library with the kernels' device-side
index checks compiled in); any other value is taken as the library's path.
"""
from __future__ import annotations

import ctypes
import sys
from pathlib import Path
from typing import Sequence

_LIB_PATH = Path(__file__).resolve().parent / "libgar.so"


def _lib_path() -> Path:
    import os
    choice = os.environ.get("GAR_LIBRARY", "")
    if choice == "":
        return _LIB_PATH
    if choice == "debug":
        return _LIB_PATH.with_name("libgar_debug.so")
    return Path(choice)

AR_OK, AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_ERR_CUDA, AR_ERR_TIMEOUT, AR_ERR_STATE, \
    AR_ERR_DEVICE_CHECK = range(7)
AR_OP_DEFAULT, AR_SUM, AR_MEAN = -1, 0, 1
AR_F32, AR_BF16 = 0, 1
AR_MAX_RANKS = 16
ELEM_BYTES = {AR_F32: 4, AR_BF16: 2}


class GarError(RuntimeError):
    """A non-OK ar_status_t from the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {ar_status_string(status)}")


class ar_bucket_t(ctypes.Structure):
    _fields_ = [("ntensors", ctypes.c_int), ("dev_ptrs", ctypes.POINTER(ctypes.c_void_p)),
                ("numel", ctypes.POINTER(ctypes.c_size_t)), ("dtype", ctypes.c_int)]


class ar_accum_t(ctypes.Structure):
    _fields_ = [("acc", ctypes.POINTER(ctypes.c_void_p)), ("scale", ctypes.c_float),
                ("first", ctypes.c_int)]


class ar_sgd_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("momentum", ctypes.c_float),
                ("master", ctypes.POINTER(ctypes.c_void_p)),
                ("momentum_buf", ctypes.POINTER(ctypes.c_void_p)),
                ("write_back_grads", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    path = _lib_path()
    if not path.exists():
        raise ImportError(f"{path} is missing: build it with "
                          "gradient_all_reduce_gb300.build.build()")
    lib = ctypes.CDLL(str(path))
    P = ctypes.c_void_p
    PP = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "ar_init": [ctypes.POINTER(P), ctypes.c_int, ctypes.c_int, ctypes.c_int],
        "ar_destroy": [P],
        "ar_all_reduce": [P, PP, PP, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, P],
        "ar_reduce_scatter": [P, PP, PP, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, P],
        "ar_all_gather": [P, PP, PP, ctypes.c_size_t, ctypes.c_int, P],
        "ar_broadcast": [P, PP, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, P],
        "ar_bucket_all_reduce": [P, ctypes.POINTER(ar_bucket_t), ctypes.c_int,
                                 ctypes.POINTER(ar_sgd_t), P],
        "ar_bucket_accumulate": [P, ctypes.POINTER(ar_bucket_t), ctypes.POINTER(ar_accum_t), P],
        "ar_bucket_all_reduce_accumulated": [P, ctypes.POINTER(ar_bucket_t),
                                             ctypes.POINTER(ar_accum_t), ctypes.c_int,
                                             ctypes.POINTER(ar_sgd_t), P],
        "ar_sharded_sgd_step": [P, PP, PP, PP, PP, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                ctypes.c_float, ctypes.c_float, P],
        "ar_syncbn_stats": [P, PP, PP, ctypes.POINTER(ctypes.c_uint64), PP, PP, ctypes.c_size_t,
                            ctypes.c_float, P],
        "ar_bucket_plan": [ctypes.c_int, ctypes.POINTER(ctypes.c_size_t), ctypes.c_size_t,
                           ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)],
        "ar_get_async_error": [P],
        "ar_selftest_wait_timeout": [P, ctypes.c_uint, P],
        "ar_reducer_create": [ctypes.POINTER(P), P, ctypes.POINTER(ar_bucket_t), ctypes.c_size_t,
                              ctypes.c_int, ctypes.POINTER(ar_sgd_t)],
        "ar_reducer_mark_ready": [P, ctypes.c_int, P],
        "ar_reducer_mark_ready_many": [P, ctypes.POINTER(ctypes.c_int), ctypes.c_int, P],
        "ar_reducer_finalize": [P, P],
        "ar_reducer_set_sgd": [P, ctypes.c_float, ctypes.c_float],
        "ar_reducer_wait_bucket": [P, ctypes.c_int, P],
        "ar_reducer_info": [P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)],
        "ar_reducer_launches": [P, ctypes.POINTER(ctypes.c_uint64)],
        "ar_reducer_destroy": [P],
        "ar_all_reduce_noalloc": [ctypes.c_int, PP, PP, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                  P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.ar_status_string.argtypes = [ctypes.c_int]
    lib.ar_status_string.restype = ctypes.c_char_p
    return lib


_HANDLE: ctypes.CDLL | None = None


def load() -> ctypes.CDLL:
    """The loaded libgar.so (loaded on first call; ImportError if missing)."""
    global _HANDLE
    if _HANDLE is None:
        _HANDLE = _load()
    return _HANDLE


def __getattr__(name):
    if name == "lib":
        return load()
    raise AttributeError(name)


def ar_status_string(status: int) -> str:
    return load().ar_status_string(int(status)).decode()


def _ok(status: int, what: str) -> None:
    if status != AR_OK:
        raise GarError(status, what)


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs) -> ctypes.Array:
    return (ctypes.c_void_p * len(xs))(*[_addr(x) for x in xs])


def _stream(stream) -> int:
    if stream is None:
        torch = sys.modules.get("torch")
        return int(torch.cuda.current_stream().cuda_stream) if torch is not None else 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def ar_init(nranks: int, cuda_device: int = 0, default_op: int = AR_MEAN) -> int:
    """Create a device group of ``nranks`` replicas; returns the comm handle."""
    comm = ctypes.c_void_p()
    _ok(load().ar_init(ctypes.byref(comm), int(nranks), int(cuda_device), int(default_op)), "ar_init")
    return int(comm.value)


def ar_destroy(comm: int) -> None:
    _ok(load().ar_destroy(comm), "ar_destroy")


def ar_all_reduce(comm: int, send: Sequence, recv: Sequence, count: int, dtype: int,
                  op: int = AR_OP_DEFAULT, stream=None) -> None:
    _ok(load().ar_all_reduce(comm, _ptr_array(send), _ptr_array(recv), int(count), int(dtype),
                          int(op), _stream(stream)), "ar_all_reduce")


def ar_all_reduce_noalloc(nranks: int, send: Sequence, recv: Sequence, count: int, dtype: int,
                          op: int, stream=None) -> None:
    """All-reduce on the current CUDA device without a comm and without any
    allocation (see include/gar.h): for callers that may not allocate
    device memory themselves."""
    _ok(load().ar_all_reduce_noalloc(int(nranks), _ptr_array(send), _ptr_array(recv), int(count),
                                     int(dtype), int(op), _stream(stream)), "ar_all_reduce_noalloc")


def ar_reduce_scatter(comm: int, send: Sequence, recv: Sequence, count: int, dtype: int,
                      op: int = AR_OP_DEFAULT, stream=None) -> None:
    _ok(load().ar_reduce_scatter(comm, _ptr_array(send), _ptr_array(recv), int(count), int(dtype),
                              int(op), _stream(stream)), "ar_reduce_scatter")


def ar_all_gather(comm: int, send: Sequence, recv: Sequence, count: int, dtype: int,
                  stream=None) -> None:
    _ok(load().ar_all_gather(comm, _ptr_array(send), _ptr_array(recv), int(count), int(dtype),
                          _stream(stream)), "ar_all_gather")


def ar_broadcast(comm: int, buf: Sequence, count: int, dtype: int, root: int = 0,
                 stream=None) -> None:
    _ok(load().ar_broadcast(comm, _ptr_array(buf), int(count), int(dtype), int(root),
                         _stream(stream)), "ar_broadcast")


def ar_bucket_all_reduce(comm: int, tensors: Sequence[Sequence], numel: Sequence[int], dtype: int,
                         op: int = AR_OP_DEFAULT, sgd=None, stream=None) -> None:
    """``tensors[t][r]`` is rank r's replica of tensor t.  ``sgd`` is None or
    (lr, momentum, master[t], momentum_buf[t], write_back_grads)."""
    flat = [x for reps in tensors for x in reps]
    ptrs = _ptr_array(flat)
    nel = (ctypes.c_size_t * max(len(numel), 1))(*[int(n) for n in numel])
    b = ar_bucket_t(len(tensors), ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                    ctypes.cast(nel, ctypes.POINTER(ctypes.c_size_t)), int(dtype))
    s = None
    if sgd is not None:
        lr, mom, master, mbuf, wb = sgd
        m, v = _ptr_array(master), _ptr_array(mbuf)
        s = ar_sgd_t(float(lr), float(mom), ctypes.cast(m, ctypes.POINTER(ctypes.c_void_p)),
                     ctypes.cast(v, ctypes.POINTER(ctypes.c_void_p)), int(bool(wb)))
    _ok(load().ar_bucket_all_reduce(comm, ctypes.byref(b), int(op),
                                 ctypes.byref(s) if s is not None else None, _stream(stream)),
        "ar_bucket_all_reduce")


def _bucket_struct(tensors, numel, dtype):
    ptrs = _ptr_array([x for reps in tensors for x in reps])
    nel = (ctypes.c_size_t * max(len(numel), 1))(*[int(n) for n in numel])
    b = ar_bucket_t(len(tensors), ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)),
                    ctypes.cast(nel, ctypes.POINTER(ctypes.c_size_t)), int(dtype))
    return b, (ptrs, nel)


def ar_bucket_accumulate(comm: int, tensors: Sequence[Sequence], numel: Sequence[int], dtype: int,
                         acc: Sequence[Sequence], scale: float, first: bool, stream=None) -> None:
    """A micro-batch before the last (no all-reduce): ``acc[t][r]`` (fp32)
    gets rank r's ``scale * tensors[t][r]`` (overwritten when ``first``)."""
    b, keep = _bucket_struct(tensors, numel, dtype)
    accp = _ptr_array([x for reps in acc for x in reps])
    a = ar_accum_t(ctypes.cast(accp, ctypes.POINTER(ctypes.c_void_p)), float(scale), int(bool(first)))
    _ok(load().ar_bucket_accumulate(comm, ctypes.byref(b), ctypes.byref(a), _stream(stream)),
        "ar_bucket_accumulate")


def ar_bucket_all_reduce_accumulated(comm: int, tensors: Sequence[Sequence], numel: Sequence[int],
                                     dtype: int, acc: Sequence[Sequence], scale: float, first: bool,
                                     op: int = AR_OP_DEFAULT, sgd=None, stream=None) -> None:
    """The last micro-batch: all-reduce of every rank's acc + scale * grad
    (optionally fused with SGD), results into the gradient replicas."""
    b, keep = _bucket_struct(tensors, numel, dtype)
    accp = _ptr_array([x for reps in acc for x in reps])
    a = ar_accum_t(ctypes.cast(accp, ctypes.POINTER(ctypes.c_void_p)), float(scale), int(bool(first)))
    s = None
    if sgd is not None:
        lr, mom, master, mbuf, wb = sgd
        m, v = _ptr_array(master), _ptr_array(mbuf)
        s = ar_sgd_t(float(lr), float(mom), ctypes.cast(m, ctypes.POINTER(ctypes.c_void_p)),
                     ctypes.cast(v, ctypes.POINTER(ctypes.c_void_p)), int(bool(wb)))
    _ok(load().ar_bucket_all_reduce_accumulated(comm, ctypes.byref(b), ctypes.byref(a), int(op),
                                                ctypes.byref(s) if s is not None else None,
                                                _stream(stream)),
        "ar_bucket_all_reduce_accumulated")


def ar_sharded_sgd_step(comm: int, grads: Sequence, params: Sequence, master_shards: Sequence,
                        momentum_shards: Sequence, count: int, dtype: int, lr: float,
                        momentum: float, op: int = AR_OP_DEFAULT, stream=None) -> None:
    """ZeRO-1 step: reduce-scatter, each owner's SGD on its fp32 shard, and
    all-gather of the updated weights into every params replica, in one pass."""
    _ok(load().ar_sharded_sgd_step(comm, _ptr_array(grads), _ptr_array(params),
                                   _ptr_array(master_shards), _ptr_array(momentum_shards),
                                   int(count), int(dtype), int(op), float(lr), float(momentum),
                                   _stream(stream)), "ar_sharded_sgd_step")


def ar_syncbn_stats(comm: int, sums: Sequence, sqsums: Sequence, counts: Sequence[int],
                    means: Sequence, invstds: Sequence, channels: int, eps: float = 1e-5,
                    stream=None) -> None:
    """Pooled batch-norm statistics for every rank from the ranks'
    per-channel sums, sums of squares and value counts."""
    cnt = (ctypes.c_uint64 * max(len(counts), 1))(*[int(c) for c in counts])
    _ok(load().ar_syncbn_stats(comm, _ptr_array(sums), _ptr_array(sqsums), cnt, _ptr_array(means),
                               _ptr_array(invstds), int(channels), float(eps), _stream(stream)),
        "ar_syncbn_stats")


def ar_bucket_plan(nbytes: Sequence[int], cap_bytes: int = 25 << 20) -> list[int]:
    """Bucket index of each tensor (registration order in; reverse-order fill)."""
    T = len(nbytes)
    nb = (ctypes.c_size_t * max(T, 1))(*[int(n) for n in nbytes])
    out = (ctypes.c_int * max(T, 1))()
    k = ctypes.c_int()
    _ok(load().ar_bucket_plan(T, nb, int(cap_bytes), out, ctypes.byref(k)), "ar_bucket_plan")
    return list(out)[:T]


def ar_selftest_wait_timeout(comm: int, timeout_ms: int = 100, stream=None) -> None:
    _ok(load().ar_selftest_wait_timeout(comm, int(timeout_ms), _stream(stream)),
        "ar_selftest_wait_timeout")


def ar_get_async_error(comm: int) -> int:
    """The comm's sticky device-side status (an ar_status_t, not raised)."""
    return int(load().ar_get_async_error(comm))


class PreparedBucket:
    """An ar_bucket_all_reduce call with its argument structures built once
    (the pointer and length arrays stay alive with this object), so that a
    training loop re-issues the same call without rebuilding them."""

    def __init__(self, comm: int, tensors: Sequence[Sequence], numel: Sequence[int], dtype: int,
                 op: int = AR_OP_DEFAULT, sgd=None):
        flat = [x for reps in tensors for x in reps]
        self._ptrs = _ptr_array(flat)
        self._nel = (ctypes.c_size_t * max(len(numel), 1))(*[int(n) for n in numel])
        self._bucket = ar_bucket_t(len(tensors), ctypes.cast(self._ptrs, ctypes.POINTER(ctypes.c_void_p)),
                                   ctypes.cast(self._nel, ctypes.POINTER(ctypes.c_size_t)), int(dtype))
        self._sgd = None
        if sgd is not None:
            lr, mom, master, mbuf, wb = sgd
            self._m, self._v = _ptr_array(master), _ptr_array(mbuf)
            self._sgd = ar_sgd_t(float(lr), float(mom),
                                 ctypes.cast(self._m, ctypes.POINTER(ctypes.c_void_p)),
                                 ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p)), int(bool(wb)))
        self._fn = load().ar_bucket_all_reduce
        self._args = (comm, ctypes.byref(self._bucket), int(op),
                      ctypes.byref(self._sgd) if self._sgd is not None else None)

    def __call__(self, stream=None) -> None:
        _ok(self._fn(*self._args, _stream(stream)), "ar_bucket_all_reduce")


class Reducer:
    """A DDP gradient reducer (``ar_reducer_*``): ``grads[t][r]`` is rank
    r's replica of tensor t, tensors in registration order.  The argument
    structures stay alive with this object, as the C side keeps only
    pointers validated at creation."""

    def __init__(self, comm: int, grads: Sequence[Sequence], numel: Sequence[int], dtype: int,
                 cap_bytes: int = 25 << 20, op: int = AR_OP_DEFAULT, sgd=None):
        flat = [x for reps in grads for x in reps]
        self._ptrs = _ptr_array(flat)
        self._nel = (ctypes.c_size_t * max(len(numel), 1))(*[int(n) for n in numel])
        self.ntensors = len(grads)
        b = ar_bucket_t(len(grads), ctypes.cast(self._ptrs, ctypes.POINTER(ctypes.c_void_p)),
                        ctypes.cast(self._nel, ctypes.POINTER(ctypes.c_size_t)), int(dtype))
        s = None
        if sgd is not None:
            lr, mom, master, mbuf, wb = sgd
            self._m, self._v = _ptr_array(master), _ptr_array(mbuf)
            s = ar_sgd_t(float(lr), float(mom), ctypes.cast(self._m, ctypes.POINTER(ctypes.c_void_p)),
                         ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p)), int(bool(wb)))
        h = ctypes.c_void_p()
        L = load()
        _ok(L.ar_reducer_create(ctypes.byref(h), comm, ctypes.byref(b), int(cap_bytes), int(op),
                                ctypes.byref(s) if s is not None else None), "ar_reducer_create")
        self.handle = int(h.value)
        self._mark = L.ar_reducer_mark_ready
        self._mark_many = L.ar_reducer_mark_ready_many
        self._finalize = L.ar_reducer_finalize

    def mark_ready(self, tensor: int, stream=None) -> None:
        _ok(self._mark(self.handle, int(tensor), _stream(stream)), "ar_reducer_mark_ready")

    def marks(self, tensors: Sequence[int]) -> ctypes.Array:
        """A list of tensor indices marshalled once, for a mark_ready_many
        call repeated every step (the library still checks every index)."""
        return (ctypes.c_int * len(tensors))(*[int(t) for t in tensors])

    def mark_ready_many(self, tensors, stream=None) -> None:
        """``tensors``: indices, or the array ``marks`` made of them."""
        arr = tensors if isinstance(tensors, ctypes.Array) else self.marks(tensors)
        _ok(self._mark_many(self.handle, arr, len(arr), _stream(stream)),
            "ar_reducer_mark_ready_many")

    def finalize(self, stream=None) -> None:
        _ok(self._finalize(self.handle, _stream(stream)), "ar_reducer_finalize")

    def wait_bucket(self, bucket: int, stream=None) -> None:
        _ok(load().ar_reducer_wait_bucket(self.handle, int(bucket), _stream(stream)),
            "ar_reducer_wait_bucket")

    def set_sgd(self, lr: float, momentum: float) -> None:
        _ok(load().ar_reducer_set_sgd(self.handle, float(lr), float(momentum)), "ar_reducer_set_sgd")

    def bucket_of(self) -> list[int]:
        k = ctypes.c_int()
        out = (ctypes.c_int * max(self.ntensors, 1))()
        _ok(load().ar_reducer_info(self.handle, ctypes.byref(k), out), "ar_reducer_info")
        return list(out)[:self.ntensors]

    def launches(self) -> int:
        """Kernel launches issued by this reducer so far."""
        k = ctypes.c_uint64()
        _ok(load().ar_reducer_launches(self.handle, ctypes.byref(k)), "ar_reducer_launches")
        return int(k.value)

    def destroy(self) -> None:
        if self.handle:
            _ok(load().ar_reducer_destroy(self.handle), "ar_reducer_destroy")
            self.handle = 0


class PreparedCall:
    """One of the flat collectives (``ar_all_reduce``, ``ar_reduce_scatter``,
    ``ar_all_gather``, ``ar_broadcast``, ``ar_sharded_sgd_step``,
    ``ar_syncbn_stats``) with its pointer arrays marshalled once, for a loop
    that repeats the same call on the same buffers: ``PreparedCall(
    "ar_all_reduce", comm, send, recv, count, dtype, op)(stream)``.  The
    library still validates every call."""

    _LAYOUT = {
        "ar_all_reduce": ("comm", "ptrs", "ptrs", "size", "int", "int"),
        "ar_reduce_scatter": ("comm", "ptrs", "ptrs", "size", "int", "int"),
        "ar_all_gather": ("comm", "ptrs", "ptrs", "size", "int"),
        "ar_broadcast": ("comm", "ptrs", "size", "int", "int"),
        "ar_sharded_sgd_step": ("comm", "ptrs", "ptrs", "ptrs", "ptrs", "size", "int", "int",
                                "float", "float"),
        "ar_syncbn_stats": ("comm", "ptrs", "ptrs", "u64s", "ptrs", "ptrs", "size", "float"),
    }

    def __init__(self, name: str, *args):
        kinds = self._LAYOUT[name]
        if len(args) != len(kinds):
            raise TypeError(f"{name} takes {len(kinds)} arguments before the stream")
        self._keep = []
        conv = []
        for kind, a in zip(kinds, args):
            if kind == "ptrs":
                arr = _ptr_array(a)
                self._keep.append(arr)
                conv.append(arr)
            elif kind == "u64s":
                arr = (ctypes.c_uint64 * max(len(a), 1))(*[int(x) for x in a])
                self._keep.append(arr)
                conv.append(arr)
            elif kind == "float":
                conv.append(float(a))
            else:
                conv.append(int(a))
        self._fn = getattr(load(), name)
        self._args = tuple(conv)
        self._name = name

    def __call__(self, stream=None) -> None:
        _ok(self._fn(*self._args, _stream(stream)), self._name)
