"""Pins of the synthetic-input module (no method arithmetic lives there)."""
import numpy as np

import workloads
from golden import lines, table


def test_splitmix64_published_outputs():
    want = [int(v, 16) for v in lines("splitmix64_seed0.txt")]
    assert [workloads.splitmix64_scalar(0, i) for i in range(4)] == want
    assert [int(v) for v in workloads.splitmix64(0, np.arange(4))] == want


def test_counter_form_matches_sequential_generator():
    """Output i of the counter form is the (i+1)-th call of the stateful
    generator: state += GOLDEN, then mix."""
    state, seed = 12345, 12345
    for i in range(50):
        state = (state + workloads.GOLDEN) & ((1 << 64) - 1)
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & ((1 << 64) - 1)
        assert workloads.splitmix64_scalar(seed, i) == z ^ (z >> 31)


def test_uniform_is_exact_and_in_range():
    u = workloads.uniform_f32(3, 1 << 16)
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    k = (u.astype(np.float64) + 1.0) * 2.0 ** 23
    assert np.array_equal(k, np.round(k))
    # drawing a slice or scattered indices gives the same values
    assert np.array_equal(workloads.uniform_f32(3, 100, start=500), u[500:600])
    idx = np.array([7, 65535, 0], dtype=np.uint64)
    assert np.array_equal(workloads.uniform_f32(3, 0, idx=idx), u[idx.astype(np.int64)])


def test_normal_moments():
    x = workloads.normal_f32(0, 1 << 20, std=0.02)
    assert abs(float(x.mean())) < 1e-4 and abs(float(x.std()) / 0.02 - 1) < 0.01


def test_bf16_inputs_truncate():
    x = np.array([1.0, -1.00390625 - 2 ** -20], np.float32)
    assert workloads.bf16_trunc(x).tolist() == [0x3F80, 0xBF80]


def test_vit_b16_shapes_match_page_count():
    g = table("vit_b16_param_count.txt")
    n = workloads.vit_b16_numels()
    assert sum(n) == int(g["params"]) == workloads.VIT_B16_PARAMS
    assert len(n) == int(g["tensors"])


def test_vit_b16_order_matches_torch_modules():
    """The shape list follows torch's registration order for the same
    modules (the model's own tensors first, then its submodules)."""
    import torch
    import torch.nn as nn

    class ViT(nn.Module):
        def __init__(self):
            super().__init__()
            D = workloads.VIT_D
            self.patch = nn.Conv2d(3, D, workloads.VIT_PATCH, stride=workloads.VIT_PATCH)
            self.cls = nn.Parameter(torch.zeros(1, 1, D))
            self.pos = nn.Parameter(torch.zeros(1, workloads.VIT_TOKENS, D))
            self.blocks = nn.ModuleList(
                nn.TransformerEncoderLayer(D, 12, workloads.VIT_MLP, norm_first=True,
                                           batch_first=True) for _ in range(workloads.VIT_LAYERS))
            self.norm = nn.LayerNorm(D)
            self.head = nn.Linear(D, workloads.VIT_CLASSES)

    with torch.device("meta"):
        m = ViT()
    got = [(n, tuple(p.shape)) for n, p in m.named_parameters()]
    assert got == workloads.vit_b16_shapes()
