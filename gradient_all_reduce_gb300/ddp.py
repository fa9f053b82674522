"""DDP-style gradient synchronisation of P model replicas on one GPU.

DDP overlaps the all-reduce with the backward pass: gradients are packed
into ~25 MB buckets in reverse parameter order, and a bucket's all-reduce
is launched as soon as all of its gradients are ready, while the backward
pass goes on ("Distributed Training", computervisiononline.com, "Data
parallelism and all-reduce"; Lecture 8, rd.me/cs336/lec8, Part 2 s.1).

``ReplicaDDP`` wires a torch module to the library's reducer
(``ar_reducer_*``): each parameter's ``.grad`` is a view into rank 0's flat
gradient buffer (ranks 1..P-1 get flat buffers of their own), and an
autograd post-accumulate hook counts the parameter's gradient as final;
when a bucket's last gradient is final, its tensors are marked ready in one
call on the current stream, so the reducer launches the bucket during the
backward pass.  (One library call per bucket instead of one per parameter:
the hooks run on the host inside the backward pass.)  ``finish()`` ends the
step.  All arithmetic runs in the library's kernels; this module only wires
buffers and hooks.
"""
from __future__ import annotations

import torch

import gradient_all_reduce_gb300 as gar

_AR_DTYPE = {torch.float32: gar.AR_F32, torch.bfloat16: gar.AR_BF16}


class ReplicaDDP:
    """P replicas of ``module``'s gradients, reduced bucket by bucket.

    ``sgd`` = (lr, momentum) fuses the SGD-momentum step on fp32 master
    weights (initialised from the module's parameters) into each bucket's
    kernel; the reduced gradient is then also written back to every
    replica.  ``hooks_enabled`` lets a caller run backward passes that do
    not mark anything (e.g. the passes of ranks other than the last)."""

    def __init__(self, comm: int, module: torch.nn.Module, P: int, cap_bytes: int = 25 << 20,
                 op: int = gar.AR_MEAN, sgd: tuple[float, float] | None = None):
        self.params = [p for p in module.parameters() if p.requires_grad]
        if not self.params:
            raise ValueError("module has no trainable parameters")
        dtype = self.params[0].dtype
        if dtype not in _AR_DTYPE or any(p.dtype != dtype for p in self.params):
            raise TypeError("all parameters must share one dtype, float32 or bfloat16")
        dev = self.params[0].device
        self.numels = [p.numel() for p in self.params]
        offs = [0]
        for n in self.numels:
            offs.append(offs[-1] + n)
        self.offs = offs
        n = offs[-1]
        # rank r's flat gradient buffer; rank 0's holds the module's .grad views
        self.flat = [torch.zeros(n, dtype=dtype, device=dev) for _ in range(P)]
        for t, p in enumerate(self.params):
            p.grad = self.flat[0][offs[t]:offs[t + 1]].view_as(p)
        grads = [[f[offs[t]:offs[t + 1]] for f in self.flat] for t in range(len(self.params))]
        sgd_args = None
        if sgd is not None:
            self.master = torch.cat([p.detach().float().reshape(-1) for p in self.params])
            self.momentum = torch.zeros(n, dtype=torch.float32, device=dev)
            sgd_args = (sgd[0], sgd[1],
                        [self.master[offs[t]:offs[t + 1]] for t in range(len(self.params))],
                        [self.momentum[offs[t]:offs[t + 1]] for t in range(len(self.params))], 1)
        self.reducer = gar.Reducer(comm, grads, self.numels, _AR_DTYPE[dtype], cap_bytes, op,
                                   sgd=sgd_args)
        self._bucket_of = self.reducer.bucket_of()
        nb = max(self._bucket_of) + 1
        self._bucket_tensors = [[] for _ in range(nb)]
        for t in range(len(self.params) - 1, -1, -1):      # the order gradients become final
            self._bucket_tensors[self._bucket_of[t]].append(t)
        self._pending = [len(ts) for ts in self._bucket_tensors]
        self._bucket_marks = [self.reducer.marks(ts) for ts in self._bucket_tensors]
        self.hooks_enabled = True
        self._stream = None          # handle of the stream the current backward runs on
        self._handles = []
        for t, p in enumerate(self.params):
            self._handles.append(p.register_post_accumulate_grad_hook(self._hook(t)))

    def _hook(self, t: int):
        b = self._bucket_of[t]

        def hook(_param):
            if self.hooks_enabled:
                if self._stream is None:   # looked up once per step
                    self._stream = torch.cuda.current_stream().cuda_stream
                self._pending[b] -= 1
                if self._pending[b] == 0:
                    self.reducer.mark_ready_many(self._bucket_marks[b], self._stream)
        return hook

    def replica_grad(self, rank: int, t: int) -> torch.Tensor:
        """Rank ``rank``'s gradient of parameter ``t`` (a view)."""
        return self.flat[rank][self.offs[t]:self.offs[t + 1]].view_as(self.params[t])

    def point_grads_at(self, rank: int) -> None:
        """Make the module's .grad tensors views of rank ``rank``'s buffer
        (to run that rank's backward pass with the same module)."""
        for t, p in enumerate(self.params):
            p.grad = self.replica_grad(rank, t)

    def zero_(self) -> None:
        for f in self.flat:
            f.zero_()

    def finish(self, stream=None) -> None:
        """End of the step: every bucket launched, the stream ordered after them."""
        self.reducer.finalize(torch.cuda.current_stream() if stream is None else stream)
        self._stream = None
        self._pending = [len(ts) for ts in self._bucket_tensors]

    def close(self) -> None:
        for h in self._handles:
            h.remove()
        self._handles = []
        self.reducer.destroy()
