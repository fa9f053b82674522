"""The host-side argument behind the kernels' bf16-only division
(div_small_bf16): for a small divisor d that is not a power of two, the
product y = RN(x * RN(1/d)) lies within a few units in the last place of the
correctly rounded quotient q = RN(x / d), so y and q round to the same bf16
unless y's low 16 bits lie next to the tie 0x8000.  Checked here with NumPy's
IEEE float32 arithmetic on a sample of inputs (the GPU test checks the device
function itself on all 2**32 inputs)."""
import numpy as np
import pytest


def _bf16_rne(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint64)
    out = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) & 0xFFFF
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x7FFFFF) != 0)
    return np.where(nan, 0x7FC0, out)


def _inputs() -> np.ndarray:
    rng = np.random.default_rng(12)
    rand = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    # every exponent with low halves around the bf16 tie, and subnormals
    hi = (np.arange(1 << 9, dtype=np.uint32) << 23)
    lo = np.array([0, 1, 2, 0x7FFB, 0x7FFC, 0x7FFF, 0x8000, 0x8001, 0x8004, 0xFFFF], np.uint32)
    mant = (rng.integers(0, 1 << 7, size=hi.size, dtype=np.uint64).astype(np.uint32) << 16)
    edge = (hi[:, None] | mant[:, None] | lo[None, :]).ravel()
    return np.concatenate([rand, edge])


@pytest.mark.parametrize("d", [3, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15])
def test_product_rounds_to_the_quotients_bf16_outside_the_window(d):
    x = _inputs().view(np.float32)
    dd = np.float32(d)
    r = np.float32(1) / dd
    with np.errstate(all="ignore"):
        q = x / dd
        y = x * r
    qb, yb = q.view(np.uint32), y.view(np.uint32)
    fin = np.isfinite(q)
    dist = np.abs(yb[fin].astype(np.int64) - qb[fin].astype(np.int64))
    assert dist.max() <= 3
    outside = ((yb - np.uint32(0x7FFC)) & np.uint32(0xFFFF)) >= 8
    assert np.array_equal(_bf16_rne(yb[outside]), _bf16_rne(qb[outside]))


def test_the_window_is_needed():
    """Inside the window the product alone would round differently at times:
    the fallback is not dead code."""
    x = _inputs().view(np.float32)
    diff = 0
    for d in (3, 5, 7, 11, 13):
        dd = np.float32(d)
        with np.errstate(all="ignore"):
            q = x / dd
            y = x * (np.float32(1) / dd)
        diff += int(np.count_nonzero(_bf16_rne(y.view(np.uint32)) != _bf16_rne(q.view(np.uint32))))
    assert diff > 0
