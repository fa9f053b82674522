"""The oracle against its pins (exact arithmetic, library routines, worked
examples and invariants): see ``pins.py``."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(oracle.lib())


def test_bf16_round_exhaustive_against_torch():
    """The oracle's fp32 -> bf16 round-to-nearest-even against torch's CPU
    cast for every one of the 2**32 fp32 bit patterns (a NaN only has to
    stay a NaN: payloads are not compared)."""
    import numpy as np
    import torch
    L = oracle.lib()
    chunk = 1 << 26
    base = np.arange(chunk, dtype=np.uint32)
    u = np.empty(chunk, np.uint32)
    for start in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(start), out=u)
        f = u.view(np.float32)
        got = oracle.f32_to_bf16(f, L=L)
        want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        bad = np.flatnonzero((got != want) & ~nan)
        assert bad.size == 0, f"x bits {int(u[bad[0]]):#010x}: {int(got[bad[0]]):#06x} != {int(want[bad[0]]):#06x}"
        g_exp, g_man = (got[nan] >> 7) & 0xFF, got[nan] & 0x7F
        assert np.all((g_exp == 0xFF) & (g_man != 0)), "a NaN did not stay a NaN"
