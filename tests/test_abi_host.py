"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point that include/gar.h declares, refuses bad arguments before
touching CUDA, and its bucket assignment equals the oracle's."""
import re
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def gar():
    from gradient_all_reduce_gb300.build import build
    build()
    import gradient_all_reduce_gb300
    return gradient_all_reduce_gb300


def declared_functions():
    text = "\n".join(p.read_text() for p in sorted((ROOT / "include").glob("*.h")))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(gar):
    names = declared_functions()
    assert "ar_all_reduce" in names and "ar_bucket_all_reduce" in names
    for name in names:
        assert hasattr(gar.lib, name), name


def test_no_oracle_or_torch_in_the_product():
    """The product path neither imports the oracle nor falls back to torch
    arithmetic: its Python sources name neither, and libgar.so exports no
    oracle symbol."""
    pkg = ROOT / "gradient_all_reduce_gb300"
    for p in pkg.glob("*.py"):
        src = p.read_text()
        assert "import oracle" not in src and "from oracle" not in src, p
    for p in (pkg / "csrc").iterdir():
        assert "oracle" not in p.read_text().lower(), p


def test_status_strings(gar):
    for s in range(6):
        assert gar.ar_status_string(s).startswith("AR_")
    assert "unknown" in gar.ar_status_string(99)


def test_refusals_without_a_gpu(gar):
    """Argument errors are reported before any CUDA call."""
    import ctypes
    comm = ctypes.c_void_p()
    assert gar.lib.ar_init(None, 2, 0, gar.AR_SUM) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_init(ctypes.byref(comm), 0, 0, gar.AR_SUM) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_init(ctypes.byref(comm), 17, 0, gar.AR_SUM) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_init(ctypes.byref(comm), 2, 0, 7) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_destroy(None) == gar.AR_ERR_STATE
    assert gar.lib.ar_all_reduce(None, None, None, 1, 0, 0, None) == gar.AR_ERR_STATE
    assert gar.lib.ar_bucket_all_reduce(None, None, 0, None, None) == gar.AR_ERR_STATE
    assert gar.lib.ar_get_async_error(None) == gar.AR_ERR_STATE
    k = ctypes.c_int()
    assert gar.lib.ar_bucket_plan(-1, None, 10, None, ctypes.byref(k)) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_bucket_plan(0, None, 0, None, ctypes.byref(k)) == gar.AR_ERR_INVALID_ARG
    assert gar.lib.ar_bucket_plan(0, None, 10, None, ctypes.byref(k)) == gar.AR_OK and k.value == 0


def test_bucket_plan_matches_oracle(gar):
    """The library's bucket assignment equals the oracle's on the ViT-B/16
    gradient set and on random size lists (integer results, bit-exact)."""
    import oracle
    import workloads
    nb = [2 * n for n in workloads.vit_b16_numels()]
    plan = gar.ar_bucket_plan(nb, 25 << 20)
    assert plan == oracle.bucket_plan(nb, 25 << 20)
    assert max(plan) + 1 == 8
    rng = np.random.default_rng(1)
    for _ in range(200):
        sizes = [int(s) for s in rng.integers(0, 100, size=int(rng.integers(0, 40)))]
        cap = int(rng.integers(1, 200))
        assert gar.ar_bucket_plan(sizes, cap) == oracle.bucket_plan(sizes, cap)
    huge = [2 ** 62, 2 ** 62, 5]
    assert gar.ar_bucket_plan(huge, 2 ** 63) == oracle.bucket_plan(huge, 2 ** 63)


def test_no_alloc_entry_point_source_allocates_nothing():
    """The allocation-free all-reduce's source file (its static array, its
    set-up and the entry point) calls no allocating CUDA routine."""
    src = (ROOT / "gradient_all_reduce_gb300" / "csrc" / "gar_noalloc.cu").read_text()
    section = src[src.index("// All-reduce without any allocation."):]
    section = re.sub(r"//[^\n]*", "", section)   # the comments explain why; check the code
    for word in ("cudaMalloc", "cudaFree", "cudaHostAlloc", "cudaMallocAsync", "new ", "malloc("):
        assert word not in section, word


def test_reducer_marks_pass_the_indices_and_their_count(gar):
    """Reducer.mark_ready_many passes the indices and their number, whether
    it gets a list or the array Reducer.marks made once (checked against a
    stand-in for the library call, no GPU)."""
    r = object.__new__(gar.Reducer)
    r.handle = 1234
    seen = []

    def call(handle, arr, n, stream):
        seen.append((handle, [arr[i] for i in range(n)], n, stream))
        return gar.AR_OK

    r._mark_many = call
    prepared = r.marks(range(5, 2, -1))
    r.mark_ready_many(prepared, 7)
    r.mark_ready_many(prepared, 7)
    r.mark_ready_many([2, 0], 7)
    r.mark_ready_many([], 7)
    assert seen == [(1234, [5, 4, 3], 3, 7), (1234, [5, 4, 3], 3, 7), (1234, [2, 0], 2, 7),
                    (1234, [], 0, 7)]
