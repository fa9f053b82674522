"""fp64 MLP gradients for the DDP-equivalence check -- TEST INFRASTRUCTURE ONLY.

The identity checked ("Distributed Training", computervisiononline.com,
"Data parallelism and all-reduce"): for a loss averaged over a batch split
into P equal shards, the mean over ranks of each shard's mean-loss gradient
is the full-batch gradient.  The page's own simulation shows the same thing
for a small CNN ("How to Apply It", part 1: 6.7e-16 in float64, 5.2e-07 in
float32); "Lecture 8 -- Parallelism" (rd.me/cs336/lec8, Part 2 s.1) runs the
DDP step on an MLP.

Network (the reading taken for "a 4-layer MLP, 1024 -> 1024, ReLU, no
bias"): h_0 = X, h_k = ReLU(h_{k-1} W_k^T) for k = 1..3, out = h_3 W_4^T;
ReLU'(0) = 0.  Loss: the mean over all B x width entries of (out - T)^2.
The backward pass is the chain rule written out, one layer at a time;
matrix products are NumPy's (a library primitive).
"""
from __future__ import annotations

import numpy as np


def forward_backward(ws, x, t):
    """Loss and dL/dW_k for every layer, all in fp64."""
    hs = [x]                      # layer inputs h_0 .. h_{K-1}
    zs = []                       # pre-activations of the hidden layers
    h = x
    K = len(ws)
    for k, w in enumerate(ws):
        z = h @ w.T
        if k < K - 1:
            zs.append(z)
            h = np.maximum(z, 0.0)
            hs.append(h)
        else:
            out = z
    diff = out - t
    loss = float(np.mean(diff * diff))
    d = 2.0 * diff / diff.size    # dL/d(out)
    grads = [None] * K
    for k in range(K - 1, -1, -1):
        grads[k] = d.T @ hs[k]    # dL/dW_k = d^T h_{k-1}
        if k > 0:
            d = (d @ ws[k]) * (zs[k - 1] > 0.0)
    return loss, grads


def shard_gradients(ws, x, t, shards: int):
    """Per-shard gradients: rows [s*B/P, (s+1)*B/P) with their own mean loss."""
    B = x.shape[0]
    if B % shards:
        raise ValueError("the batch must split into equal shards")
    m = B // shards
    return [forward_backward(ws, x[s * m:(s + 1) * m], t[s * m:(s + 1) * m])[1]
            for s in range(shards)]


def linf_rel(approx, exact) -> float:
    """max |approx - exact| / max |exact| over all tensors jointly."""
    num = max(float(np.max(np.abs(np.asarray(a, np.float64) - e))) for a, e in zip(approx, exact))
    den = max(float(np.max(np.abs(e))) for e in exact)
    return num / den
