"""Seeded synthetic inputs and workload shapes, shared by the oracle tests,
the CUDA-path tests and the benchmark.

This module holds none of the all-reduce method's arithmetic. It only
draws random numbers and describes tensor shapes:

* ``splitmix64`` -- the SplitMix64 generator of Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators" (OOPSLA 2014), in its
  counter form: output ``i`` of the stream seeded with ``seed`` is
  ``mix64(seed + (i + 1) * GOLDEN)``, the value the sequential generator
  returns on its ``(i+1)``-th call.  Being counter-based, any element can be
  drawn on its own, on the host or on the GPU (``workloads/synth.cu``), with
  identical bits.
* ``uniform_f32`` -- U(-1, 1): the top 24 bits ``u`` of a draw give
  ``u * 2**-23 - 1``, exact in fp32.
* ``normal_f32`` -- an integer-exact bell-shaped draw with mean 0 and a given
  standard deviation: the sum of the four 16-bit fields of one draw
  (Irwin-Hall with four terms), centred and scaled in one fp64 multiply,
  then rounded once to fp32.  Host and device therefore produce the same
  bytes without any transcendental function.
* ``bf16_trunc`` -- bf16 inputs are the upper 16 bits of the fp32 draw
  (truncation), which is deliberately not the method's round-to-nearest
  cast.

Shapes: the ViT-B/16 gradient set of the "Distributed Training" page
(computervisiononline.com, "How to Apply It", part 3: patch embedding,
class token, position embedding, 12 pre-norm encoder blocks, final
LayerNorm, 1000-way head; 86,567,656 parameters), and the 4-layer
1024-wide MLP of the DDP-equivalence workload.
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# Irwin-Hall(4) over 16-bit fields: mean 4 * 65535 / 2, variance
# 4 * (65536**2 - 1) / 12.
IH4_MEAN = 131070
IH4_STD = float(np.sqrt((65536.0 ** 2 - 1.0) / 3.0))


def splitmix64_scalar(seed: int, i: int) -> int:
    """Output ``i`` (0-based) of SplitMix64 seeded with ``seed`` (pure Python)."""
    z = (seed + (i + 1) * GOLDEN) & _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """Vectorised ``splitmix64_scalar`` over a uint64 index array."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK) + (idx + np.uint64(1)) * np.uint64(GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def _index(start: int, n: int) -> np.ndarray:
    return np.arange(start, start + n, dtype=np.uint64)


def uniform_f32(seed: int, n: int, start: int = 0, idx: np.ndarray | None = None) -> np.ndarray:
    """U(-1,1) fp32 draws ``start .. start+n-1`` (or at ``idx``) of stream ``seed``."""
    z = splitmix64(seed, _index(start, n) if idx is None else idx)
    u = (z >> np.uint64(40)).astype(np.int64)
    return (u.astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)


def normal_scale(std: float) -> float:
    """The fp64 factor that maps a centred Irwin-Hall(4) sum to std ``std``."""
    return float(std) / IH4_STD


def normal_f32(seed: int, n: int, std: float = 1.0, start: int = 0,
               idx: np.ndarray | None = None) -> np.ndarray:
    """Bell-shaped fp32 draws with mean 0 and standard deviation ``std``."""
    z = splitmix64(seed, _index(start, n) if idx is None else idx)
    m = np.uint64(0xFFFF)
    s = ((z & m) + ((z >> np.uint64(16)) & m) + ((z >> np.uint64(32)) & m)
         + (z >> np.uint64(48))).astype(np.int64) - IH4_MEAN
    return (s.astype(np.float64) * normal_scale(std)).astype(np.float32)


def bf16_trunc(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) holding the upper half of each fp32 value."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def replica_values(kind: str, dtype: str, seed: int, n: int, std: float = 1.0,
                   start: int = 0, idx: np.ndarray | None = None) -> np.ndarray:
    """One replica's input: ``kind`` 'uniform' or 'normal'; ``dtype`` 'f32'
    (float32 array) or 'bf16' (uint16 bit patterns)."""
    if kind == "uniform":
        x = uniform_f32(seed, n, start=start, idx=idx)
    elif kind == "normal":
        x = normal_f32(seed, n, std=std, start=start, idx=idx)
    else:
        raise ValueError(kind)
    return x if dtype == "f32" else bf16_trunc(x)


# ---------------------------------------------------------------- shapes

VIT_D, VIT_LAYERS, VIT_MLP, VIT_PATCH, VIT_CLASSES, VIT_TOKENS = 768, 12, 3072, 16, 1000, 197
VIT_B16_PARAMS = 86_567_656  # printed on the page (part 3 output)


def vit_b16_shapes() -> list[tuple[str, tuple[int, ...]]]:
    """(name, shape) of every ViT-B/16 parameter in module registration order:
    the model's own tensors (class token, position embedding), then the patch
    convolution, the 12 encoder blocks, the final LayerNorm and the head."""
    D, L, M, P, C, T = VIT_D, VIT_LAYERS, VIT_MLP, VIT_PATCH, VIT_CLASSES, VIT_TOKENS
    out: list[tuple[str, tuple[int, ...]]] = [
        ("cls", (1, 1, D)), ("pos", (1, T, D)),
        ("patch.weight", (D, 3, P, P)), ("patch.bias", (D,)),
    ]
    for b in range(L):
        pre = f"blocks.{b}."
        out += [
            (pre + "self_attn.in_proj_weight", (3 * D, D)),
            (pre + "self_attn.in_proj_bias", (3 * D,)),
            (pre + "self_attn.out_proj.weight", (D, D)),
            (pre + "self_attn.out_proj.bias", (D,)),
            (pre + "linear1.weight", (M, D)), (pre + "linear1.bias", (M,)),
            (pre + "linear2.weight", (D, M)), (pre + "linear2.bias", (D,)),
            (pre + "norm1.weight", (D,)), (pre + "norm1.bias", (D,)),
            (pre + "norm2.weight", (D,)), (pre + "norm2.bias", (D,)),
        ]
    out += [("norm.weight", (D,)), ("norm.bias", (D,)),
            ("head.weight", (C, D)), ("head.bias", (C,))]
    return out


def vit_b16_numels() -> list[int]:
    return [int(np.prod(s)) for _, s in vit_b16_shapes()]


# DDP-equivalence MLP: 4 bias-free 1024 -> 1024 layers, batch 1024 split in 8.
MLP_WIDTH, MLP_LAYERS, MLP_BATCH, MLP_SHARDS = 1024, 4, 1024, 8
MLP_SEED_W, MLP_SEED_X, MLP_SEED_T = 0, 1, 2


def mlp_problem(width: int = MLP_WIDTH, layers: int = MLP_LAYERS, batch: int = MLP_BATCH):
    """Weights W_k (width x width, variance 1/width), inputs X and targets T
    (std 1), all fp64 arrays built from fp32 draws."""
    ws = []
    for k in range(layers):
        w = normal_f32(MLP_SEED_W, width * width, std=width ** -0.5, start=k * width * width)
        ws.append(w.astype(np.float64).reshape(width, width))
    x = normal_f32(MLP_SEED_X, batch * width).astype(np.float64).reshape(batch, width)
    t = normal_f32(MLP_SEED_T, batch * width).astype(np.float64).reshape(batch, width)
    return ws, x, t


# Seeds of the ViT-B workload: gradients of replica r use 100 + r, the fp32
# master weights use 200.
VIT_GRAD_SEED, VIT_MASTER_SEED, VIT_GRAD_STD, VIT_MASTER_STD = 100, 200, 1e-3, 0.02
