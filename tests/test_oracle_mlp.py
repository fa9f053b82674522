"""The fp64 MLP oracle and the DDP-equivalence identity.

Pins: torch.autograd in fp64 (a library routine), central finite
differences (brute force), the identity "mean of equal-shard gradients =
full-batch gradient" in fp64 at the page's round-off scale, and the exact
factor P of an undivided accumulation ("Distributed Training",
computervisiononline.com, "How to Apply It", part 1 output).
"""
import numpy as np

import oracle
import workloads
from golden import table
from oracle import mlp


def _small(width=24, batch=16, layers=4, seed=11):
    rng = np.random.default_rng(seed)
    ws = [rng.normal(0, width ** -0.5, (width, width)) for _ in range(layers)]
    return ws, rng.normal(0, 1, (batch, width)), rng.normal(0, 1, (batch, width))


def test_mlp_matches_torch_autograd():
    import torch
    ws, x, t = _small()
    loss, grads = mlp.forward_backward(ws, x, t)
    tw = [torch.tensor(w, requires_grad=True) for w in ws]
    h = torch.tensor(x)
    for k, w in enumerate(tw):
        h = h @ w.T
        if k < len(tw) - 1:
            h = torch.relu(h)
    tl = torch.mean((h - torch.tensor(t)) ** 2)
    tl.backward()
    assert abs(loss - tl.item()) <= 1e-13 * abs(loss)
    for g, w in zip(grads, tw):
        np.testing.assert_allclose(g, w.grad.numpy(), rtol=1e-11, atol=1e-15)


def test_mlp_matches_finite_differences():
    ws, x, t = _small(width=4, batch=6, seed=12)
    _, grads = mlp.forward_backward(ws, x, t)
    h = 1e-6
    for k in range(len(ws)):
        for (i, j) in [(0, 0), (1, 3), (3, 2)]:
            wp = [w.copy() for w in ws]
            wm = [w.copy() for w in ws]
            wp[k][i, j] += h
            wm[k][i, j] -= h
            fd = (mlp.forward_backward(wp, x, t)[0] - mlp.forward_backward(wm, x, t)[0]) / (2 * h)
            assert abs(fd - grads[k][i, j]) <= 1e-7 * max(1.0, abs(fd)), (k, i, j)


def test_ddp_identity_fp64():
    """Mean over 4 equal shards of the shard gradients equals the full-batch
    gradient to fp64 round-off (the page prints 6.7e-16 for its CNN)."""
    ws, x, t = _small(width=32, batch=32, seed=13)
    full = mlp.forward_backward(ws, x, t)[1]
    shards = mlp.shard_gradients(ws, x, t, 4)
    mean = [sum(s[k] for s in shards) / 4 for k in range(len(ws))]
    page = float(table("ddp_equivalence.txt")["f64"])
    assert mlp.linf_rel(mean, full) <= 100 * page


def test_undivided_accumulation_is_exactly_p_times():
    """Summing shard gradients without dividing gives P times the full-batch
    gradient (the page prints a norm ratio of 4.000000000000 for P = 4)."""
    ws, x, t = _small(width=16, batch=16, seed=14)
    P = int(table("ddp_equivalence.txt")["undivided_accumulation_factor"])
    full = mlp.forward_backward(ws, x, t)[1]
    acc = [sum(s[k] for s in mlp.shard_gradients(ws, x, t, P)) for k in range(len(ws))]
    ratio = np.sqrt(sum(np.sum(a * a) for a in acc)) / np.sqrt(sum(np.sum(g * g) for g in full))
    assert abs(ratio - P) <= 1e-12 * P


def test_ddp_equivalence_full_size_oracle():
    """The DDP-equivalence workload at full size on the host: 4 layers of
    1024 x 1024, batch 1024 in 8 shards; the oracle's fp32 Mean of the
    fp32-rounded shard gradients (one 16 MiB bucket) is within the 1e-5
    L-inf/L-inf acceptance bound of the fp64 full-batch gradient."""
    ws, x, t = workloads.mlp_problem()
    full = mlp.forward_backward(ws, x, t)[1]
    shards = mlp.shard_gradients(ws, x, t, workloads.MLP_SHARDS)
    tensors = [[np.ascontiguousarray(s[k], dtype=np.float32).ravel() for s in shards]
               for k in range(len(ws))]
    assert sum(reps[0].nbytes for reps in tensors) == 16 << 20
    oracle.bucket_all_reduce(tensors, op=oracle.MEAN)
    mean = [reps[0].reshape(full[k].shape) for k, reps in enumerate(tensors)]
    err = mlp.linf_rel(mean, full)
    assert err <= float(table("ddp_equivalence.txt")["accept"]), err
    for reps in tensors:                       # every replica holds the same mean
        for r in range(1, len(reps)):
            assert np.array_equal(reps[r], reps[0])


def _micro_grads(ws, x, t, P, M):
    """grads[m][k][r]: micro-batch m of rank r (rows split rank-major, then
    into M equal micro-batches), each with its own mean loss."""
    B = x.shape[0]
    rows = B // (P * M)
    out = []
    for m in range(M):
        per_rank = []
        for r in range(P):
            lo = (r * M + m) * rows
            per_rank.append(mlp.forward_backward(ws, x[lo:lo + rows], t[lo:lo + rows])[1])
        out.append([[per_rank[r][k] for r in range(P)] for k in range(len(ws))])
    return out


def test_accumulation_and_ddp_identity_fp64():
    """P ranks x M micro-batches (loss / M each) reproduce the full-batch
    gradient to fp64 round-off (the page prints 6.7e-16 for accumulation)."""
    ws, x, t = _small(width=24, batch=32, seed=15)
    P, M = 4, 2
    full = mlp.forward_backward(ws, x, t)[1]
    grads = _micro_grads(ws, x, t, P, M)
    got = [sum(sum(grads[m][k][r] / M for m in range(M)) for r in range(P)) / P
           for k in range(len(ws))]
    assert mlp.linf_rel(got, full) <= 100 * float(table("ddp_equivalence.txt")["f64"])


def test_accumulation_full_size_oracle():
    """The DDP-equivalence MLP with each of the 8 ranks' 128 rows split into
    2 micro-batches of 64: fp32 gradients accumulated with scale 1/2 and
    all-reduced (Mean) on the last micro-batch by the oracle are within the
    1e-5 acceptance bound of the fp64 full-batch gradient."""
    ws, x, t = workloads.mlp_problem()
    P, M = workloads.MLP_SHARDS, 2
    full = mlp.forward_backward(ws, x, t)[1]
    grads = _micro_grads(ws, x, t, P, M)
    g32 = [[[np.ascontiguousarray(a, dtype=np.float32).ravel() for a in reps] for reps in gm]
           for gm in grads]
    acc = [[np.zeros(a.size, np.float32) for a in reps] for reps in g32[0]]
    oracle.bucket_accumulate(g32[0], acc, 0.5, True)
    oracle.bucket_all_reduce_accumulated(g32[1], acc, 0.5, False, op=oracle.MEAN)
    got = [g32[1][k][0].reshape(full[k].shape) for k in range(len(ws))]
    err = mlp.linf_rel(got, full)
    assert err <= float(table("ddp_equivalence.txt")["accept"]), err
