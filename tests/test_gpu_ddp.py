"""DDP-style synchronisation driven by autograd hooks (gradient_all_reduce_gb300.ddp):
the 4-layer 1024-wide MLP of the DDP-equivalence workload, P=8 replicas
(one backward pass per rank's shard on the same module), buckets launched by
the reducer while the last rank's backward pass runs."""
import numpy as np
import pytest
import torch

import gradient_all_reduce_gb300 as gar
import oracle
import workloads
from gpucase import assert_bits_equal, bits_equal_device
from golden import table
from gradient_all_reduce_gb300.ddp import ReplicaDDP
from oracle import mlp

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    yield
    torch.backends.cuda.matmul.allow_tf32 = tf32


def _mlp(ws):
    layers = []
    for k, w in enumerate(ws):
        lin = torch.nn.Linear(w.shape[1], w.shape[0], bias=False)
        with torch.no_grad():
            lin.weight.copy_(torch.from_numpy(w.astype(np.float32)))
        layers.append(lin)
        if k < len(ws) - 1:
            layers.append(torch.nn.ReLU())
    return torch.nn.Sequential(*layers).cuda()


def _shards(x, t, P):
    m = x.shape[0] // P
    xs = torch.from_numpy(x.astype(np.float32)).cuda()
    ts = torch.from_numpy(t.astype(np.float32)).cuda()
    return [(xs[r * m:(r + 1) * m], ts[r * m:(r + 1) * m]) for r in range(P)]


def test_hooks_launch_buckets_during_backward_bit_exact():
    """Snapshots of every rank's gradient, taken on the producing stream
    right before each mark, reduced by the oracle, equal the reducer's
    in-place result bit for bit (16 MiB in 2 buckets of 8 MiB)."""
    P = workloads.MLP_SHARDS
    ws, x, t = workloads.mlp_problem()
    model = _mlp(ws)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    ddp = ReplicaDDP(comm, model, P, cap_bytes=8 << 20)
    ddp.hooks_enabled = False
    snaps = [[None] * P for _ in ddp.params]
    handles = []

    def hook(tt):
        def f(_p):
            snaps[tt][P - 1] = ddp.replica_grad(P - 1, tt).detach().clone()
            ddp.reducer.mark_ready(tt, torch.cuda.current_stream())
        return f

    try:
        assert len(set(ddp.reducer.bucket_of())) == 2
        ddp.zero_()
        for r, (xr, tr) in enumerate(_shards(x, t, P)):
            ddp.point_grads_at(r)
            if r == P - 1:
                handles = [p.register_post_accumulate_grad_hook(hook(k))
                           for k, p in enumerate(ddp.params)]
            torch.nn.functional.mse_loss(model(xr), tr).backward()
            if r < P - 1:
                for k in range(len(ddp.params)):
                    snaps[k][r] = ddp.replica_grad(r, k).detach().clone()
        ddp.finish()
        torch.cuda.synchronize()
        got = [ddp.replica_grad(3, k).cpu().numpy().ravel() for k in range(len(ddp.params))]
    finally:
        for h in handles:
            h.remove()
        ddp.close()
        gar.ar_destroy(comm)
    host = [[s.cpu().numpy().ravel() for s in snaps[k]] for k in range(len(snaps))]
    oracle.bucket_all_reduce(host, op=oracle.MEAN)
    for k in range(len(host)):
        assert_bits_equal(got[k], host[k][3], f"layer {k}")


def test_replica_ddp_equals_full_batch_gradient():
    """Through ReplicaDDP's own hooks: the reduced gradient of the 8 shards
    equals the fp64 full-batch gradient within 1e-5 (L-inf/L-inf)."""
    P = workloads.MLP_SHARDS
    ws, x, t = workloads.mlp_problem()
    full = mlp.forward_backward(ws, x, t)[1]
    model = _mlp(ws)
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    ddp = ReplicaDDP(comm, model, P)
    try:
        ddp.zero_()
        for r, (xr, tr) in enumerate(_shards(x, t, P)):
            ddp.point_grads_at(r)
            ddp.hooks_enabled = r == P - 1
            torch.nn.functional.mse_loss(model(xr), tr).backward()
        ddp.finish()
        torch.cuda.synchronize()
        got = [ddp.replica_grad(0, k).double().cpu().numpy() for k in range(len(ddp.params))]
    finally:
        ddp.close()
        gar.ar_destroy(comm)
    err = mlp.linf_rel(got, full)
    assert err <= float(table("ddp_equivalence.txt")["accept"]), err


def test_replica_ddp_unused_parameter_and_two_steps():
    """A parameter that gets no gradient never completes its bucket in the
    hooks; finish() launches that bucket all the same.  Both ranks see the
    same shard, so the Mean equals one rank's gradient bit for bit (and the
    unused parameter's stays zero); two steps in a row check that the
    per-bucket counts reset."""
    torch.manual_seed(5)

    class Net(torch.nn.Module):
        def __init__(self):
            super().__init__()
            self.a = torch.nn.Linear(64, 64, bias=False)
            self.unused = torch.nn.Linear(64, 64, bias=False)
            self.b = torch.nn.Linear(64, 8)

        def forward(self, x):
            return self.b(torch.relu(self.a(x)))

    model = Net().cuda()
    ref = Net().cuda()
    ref.load_state_dict(model.state_dict())
    P = 2
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    ddp = ReplicaDDP(comm, model, P, cap_bytes=1)       # one bucket per parameter
    try:
        assert len(set(ddp.reducer.bucket_of())) == len(ddp.params)
        x = torch.randn(32, 64, device="cuda")
        for step in range(2):
            ddp.zero_()
            for r in (1, 0):
                ddp.point_grads_at(r)
                ddp.hooks_enabled = r == 0
                model(x).square().mean().backward()
            ddp.finish()
            torch.cuda.synchronize()
            assert gar.ar_get_async_error(comm) == gar.AR_OK
            ref.zero_grad(set_to_none=False)
            ref(x).square().mean().backward()
            for (name, pr), t in zip(ref.named_parameters(), range(len(ddp.params))):
                got = ddp.replica_grad(0, t)
                want = pr.grad if pr.grad is not None else torch.zeros_like(pr)
                assert bits_equal_device(got, want), (step, name)
                assert bits_equal_device(ddp.replica_grad(1, t), want), (step, name)
    finally:
        ddp.close()
        gar.ar_destroy(comm)
