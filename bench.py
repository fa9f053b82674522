"""Benchmark of the gradient all-reduce hot path on GB300.

One step is the data-parallel gradient synchronisation and optimizer step
of ViT-B/16: P = 8 replicas of the model's 86,567,656 bf16 gradients
(152 tensors in module order), packed into 25 MiB buckets in reverse
order (8 buckets), all-reduced with Mean fused with SGD (momentum 0.9, lr
0.1) on fp32 master weights, the reduced gradient written back to every
replica.  The step runs through the reducer, which launches buckets as
they complete; here every gradient is marked ready in one call, so the 8
buckets go out as one combined launch.  Throughput is algorithmic bytes
per second: per step every replica is read and written once (2*P*N*2
bytes) and the fp32 weights and momentum are read and written once (16*N
bytes), 4.155 GB in all.

Output: one JSON line (rank 0).  ``value`` times the device-resident step
with CUDA events; ``e2e`` times the same step through the public API from
pinned host buffers (gradients in, updated weights out); ``roofline``
relates the step kernel's event-timed average launch duration (the one
launch the reducer issues for all 8 buckets) to the measured HBM copy
bandwidth; ``sweep`` gives the flat all-reduce (and RS/AG/BC) GB/s
against message size for P = 2, 4, 8; ``cpu_baseline`` times the CPU
oracle on a bounded sample of the same step.

``--impl reference`` times the CPU oracle (the only reference this
project has) on the same workload and prints the same line with
"impl": "reference".

Under torchrun each rank runs its own replica group on its own GPU
(replicas only: the method runs on one GPU and has no exchange between
GPUs); the elapsed time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "all-reduce algorithm GB/s and % of GB300 HBM roofline vs bytes, P=2/4/8"
WORKLOAD = ("vit_b16_ddp_step: P=8 replicas x 86,567,656 bf16 grads, 8 x 25 MiB buckets, "
            "Mean all-reduce fused with SGD momentum (fp32 master), write-back")
P_VIT = 8
CAP = 25 << 20
# Sources of the roofline kernel and of the host code that builds its launch
# (segment table, combined launch): a committed DRAM figure holds only while
# these hash to the value recorded when it was captured.
KERNEL_SOURCES = ["gar_device.cuh", "gar_kernels.cuh", "gar_launch.h", "gar_reduce.inc",
                  "gar_reducer.cu", "gar_api.cu", "gar_host.h"]


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gar", "reference"], default="gar")
    ap.add_argument("--ref-budget", type=float, default=60.0, metavar="S",
                    help="--impl reference: seconds of oracle work the timed and warm-up steps "
                         "may take together; a step covers as much of the workload as fits")
    ap.add_argument("--no-sweep", action="store_true", help="skip the size/replica sweep")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--overlap", action="store_true",
                    help="measure the all-reduce hidden behind a ViT-B/16 backward pass instead")
    ap.add_argument("--batch", type=int, default=64, help="images per backward pass (--overlap)")
    ap.add_argument("--sweep", action="store_true",
                    help="the full size/replica sweep instead: all-reduce (Sum, Mean) and "
                         "broadcast, 4 KiB .. 1 GiB per replica, P = 2, 4, 8, fp32 and bf16")
    ap.add_argument("--case", choices=["ar", "rs", "ag", "bc", "tiny", "zero1", "sgd", "accfirst",
                                       "acc", "acclast", "syncbn"],
                    help="time one collective alone (P=8, 256 MiB per replica; ViT-sized for "
                         "zero1; one 25 MiB bf16 bucket for sgd, the bucket step with Mean + SGD, "
                         "accfirst, the first micro-batch, acc, a later one before the last, and "
                         "acclast, the last one fused with Mean + SGD; tiny is ar at P=4, 4 MiB "
                         "fp32 per replica, Mean) and print its GB/s; for profiling single kernels")
    ap.add_argument("--case-ranks", type=int, default=8, choices=range(2, 17), metavar="P",
                    help="P (2..16) for --case ar/rs/ag/bc/sgd/accfirst/acc/acclast")
    ap.add_argument("--case-dtype", choices=["f32", "bf16"], default="f32",
                    help="element type for --case ar/rs/ag/bc")
    ap.add_argument("--case-mib", type=int, default=256,
                    help="MiB per replica for --case ar/rs/ag/bc (4096: the 2**30-element fp32 "
                         "replicas of the large-bucket workload)")
    ap.add_argument("--case-op", choices=["sum", "mean"],
                    help="reduction of --case ar/rs (default: Mean for ar, Sum for rs)")
    return ap.parse_args()


# ------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity when alone)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.samples.append(parts)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for s in self.samples for k in range(4)
                          if s[4 + k].lower() == "active"})
        under_load = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(under_load) if under_load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# ------------------------------------------------------------- workloads

def vit_layout():
    import gradient_all_reduce_gb300 as gar
    import workloads
    numels = workloads.vit_b16_numels()
    plan = gar.ar_bucket_plan([2 * n for n in numels], CAP)
    offs = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
    buckets = [[] for _ in range(max(plan) + 1)]
    for t in range(len(numels) - 1, -1, -1):
        buckets[plan[t]].append(t)
    return numels, offs, buckets


def vit_bytes(n: int, P: int = P_VIT) -> int:
    return 2 * P * n * 2 + 16 * n


def vit_config(world: int) -> dict:
    """The ``config`` of the ViT step's line (both arms print the same)."""
    import workloads
    return {"workload": WORKLOAD, "P": P_VIT, "params": sum(workloads.vit_b16_numels()),
            "buckets": 8, "bucket_cap_mib": 25, "grad_dtype": "bf16", "accumulate": "fp32",
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (4.155 GB moved per step, no flush)"}


class VitStep:
    """Device buffers and prepared bucket calls of one ViT-B/16 step."""

    def __init__(self, comm, device):
        import torch
        import gradient_all_reduce_gb300 as gar
        import workloads
        from workloads import gpu as wgpu
        self.numels, self.offs, self.buckets = vit_layout()
        n = int(self.offs[-1])
        self.n = n
        self.grads = []
        for r in range(P_VIT):
            g = torch.empty(n, dtype=torch.bfloat16, device=device)
            wgpu.fill(g, "normal", workloads.VIT_GRAD_SEED + r, std=workloads.VIT_GRAD_STD)
            self.grads.append(g)
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        wgpu.fill(self.w, "normal", workloads.VIT_MASTER_SEED, std=workloads.VIT_MASTER_STD)
        self.v = torch.zeros(n, dtype=torch.float32, device=device)
        o = self.offs
        self.calls, self.bucket_bytes = [], []
        for b in self.buckets:
            ts = [[g[o[t]:o[t + 1]] for g in self.grads] for t in b]
            sgd = (0.1, 0.9, [self.w[o[t]:o[t + 1]] for t in b],
                   [self.v[o[t]:o[t + 1]] for t in b], 1)
            self.calls.append(gar.PreparedBucket(comm, ts, [self.numels[t] for t in b],
                                                 gar.AR_BF16, gar.AR_MEAN, sgd))
            self.bucket_bytes.append(vit_bytes(sum(self.numels[t] for t in b)))
        self.step_bytes = vit_bytes(n)
        # The whole step as one bucket call over all tensors in the reducer's
        # launch order (bucket by bucket, each in reverse registration order):
        # the combined launch the reducer issues when all buckets complete
        # in one call, issued directly on the caller's stream.
        order = [t for b in self.buckets for t in b]
        self.combined = gar.PreparedBucket(
            comm, [[g[o[t]:o[t + 1]] for g in self.grads] for t in order],
            [self.numels[t] for t in order], gar.AR_BF16, gar.AR_MEAN,
            (0.1, 0.9, [self.w[o[t]:o[t + 1]] for t in order],
             [self.v[o[t]:o[t + 1]] for t in order], 1))
        self.reducer = gar.Reducer(
            comm, [[g[o[t]:o[t + 1]] for g in self.grads] for t in range(len(self.numels))],
            self.numels, gar.AR_BF16, CAP, gar.AR_MEAN,
            sgd=(0.1, 0.9, [self.w[o[t]:o[t + 1]] for t in range(len(self.numels))],
                 [self.v[o[t]:o[t + 1]] for t in range(len(self.numels))], 1))
        self.reverse = self.reducer.marks(range(len(self.numels) - 1, -1, -1))

    def step(self, stream):
        """One step through the reducer: every gradient marked ready in
        reverse registration order (as a backward pass produces them; each
        bucket launches as soon as its last tensor is marked), then the step
        is finalized on the caller's stream."""
        self.reducer.mark_ready_many(self.reverse, stream)
        self.reducer.finalize(stream)

    def step_serial(self, stream):
        """The same step as eight ar_bucket_all_reduce calls on one stream."""
        for c in self.calls:
            c(stream)

    def step_combined(self, stream):
        """The same step as one ar_bucket_all_reduce call over every tensor."""
        self.combined(stream)

    def close(self):
        self.reducer.destroy()


def kernel_source_sha() -> str:
    """sha256[:16] of the bucket kernel's sources with comments and blank
    space removed: an edit that changes no code keeps the committed ncu
    figures valid, any change of code does not."""
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        text = (ROOT / "gradient_all_reduce_gb300" / "csrc" / name).read_text()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def committed_traffic():
    """DRAM bytes per launch of the roofline kernel (the combined launch of
    the ViT step) from the committed ncu summary, if it was taken on the
    current kernel source."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    if d.get("kernel_source_sha") != kernel_source_sha() or "dram_bytes_per_launch" not in d:
        return None
    return d


# ------------------------------------------------------------- GPU timing

def time_vit(args, device, stream, world):
    """K timed steps of the ViT workload through the reducer (the headline
    value).  Then, for the roofline, K steps of the kernel the reducer
    launches there (one combined launch of all 8 buckets) issued back to
    back on the timing stream; and, for comparison, K steps of the 8 bucket
    calls one after another, without and with an event pair around each."""
    import torch
    import gradient_all_reduce_gb300 as gar
    comm = gar.ar_init(P_VIT, device.index, gar.AR_MEAN)
    vs = None

    def region(fn):
        """K calls of fn back to back under one event pair.  One untimed call
        is queued first, so the timed calls find the GPU busy: the host's
        time to issue the first call, with the GPU idle, is not counted as
        kernel time."""
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn(stream)
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fn(stream)
            e0.record(stream)
            for _ in range(K):
                fn(stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / 1e3

    try:
        vs = VitStep(comm, device)
        K = args.steps
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # The clock sampler starts first (it takes a moment to produce
        # samples), so that the warm-up steps, not an idle GPU, come right
        # before the timed region.
        with ClockSampler(device.index) as clocks, torch.cuda.stream(stream):
            for _ in range(args.warmup):
                vs.step(stream)
            torch.cuda.synchronize(device)
            barrier(world)
            torch.cuda.synchronize(device)
            launches0 = vs.reducer.launches()
            start.record(stream)
            for _ in range(K):
                vs.step(stream)
            stop.record(stream)
            torch.cuda.synchronize(device)
        elapsed = start.elapsed_time(stop) / 1e3
        launches = vs.reducer.launches() - launches0
        # Host time to issue one step, on a burst short enough that the
        # launch queue never fills (a full queue makes the host wait).
        with torch.cuda.stream(stream):
            h0 = time.perf_counter()
            for _ in range(8):
                vs.step(stream)
            host_s = (time.perf_counter() - h0) * K / 8
            torch.cuda.synchronize(device)

        # The kernel roofline: the combined launch, K times back to back on
        # the timing stream.  Only this kernel runs there, and a launch's
        # CTAs wait for the previous launch to complete before they touch
        # memory, so the region's time over K is the kernel's average launch
        # duration, gaps between launches included.
        combined_s = region(vs.step_combined)
        # The 8 bucket calls one after another (per-bucket launches), and the
        # same with an event pair around each launch (each record is a
        # serialisation point of its own).
        nb = len(vs.calls)
        serial_s = region(vs.step_serial)
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nb)] for _ in range(K)]
        with torch.cuda.stream(stream):
            for k in range(K):
                for b, c in enumerate(vs.calls):
                    ev[k][b][0].record(stream)
                    c(stream)
                    ev[k][b][1].record(stream)
            torch.cuda.synchronize(device)
        launch_s = sum(e0.elapsed_time(e1) for row in ev for e0, e1 in row) / 1e3
        status = gar.ar_get_async_error(comm)
        if status != gar.AR_OK:
            raise RuntimeError(f"device status {gar.ar_status_string(status)}")
        return {"elapsed": elapsed, "launch_s": launch_s, "serial_s": serial_s,
                "combined_s": combined_s, "launches": launches, "serial_launches": K * nb,
                "step_bytes": vs.step_bytes, "launch_bytes": sum(vs.bucket_bytes) * K,
                "clocks": clocks.summary(), "n": vs.n, "host_us_per_step": host_s / K * 1e6,
                "serial_ms_per_step": serial_s / K * 1e3,
                "combined_ms_per_step": combined_s / K * 1e3}
    finally:
        if vs is not None:
            vs.close()
        gar.ar_destroy(comm)


class E2EStep:
    """The ViT step from pinned host buffers, through the public API: each
    bucket's gradient replicas are copied in (one copy per replica, spread
    over four copy streams) and its tensors marked ready on the copy
    streams, so bucket b's kernel runs while bucket b+1 is still crossing
    the host link; each bucket's updated fp32 master weights are copied out
    to ``host_w`` as soon as its kernel is done.  Bytes per step: the P
    bf16 gradient replicas in, the weights out.

    Consecutive steps are ordered per bucket, so the host link never idles
    at a step boundary: a bucket's next copy-in waits only for its previous
    kernel (which read those gradients), and its next kernel only for its
    previous copy-out (which read those weights)."""

    def __init__(self, vs, device):
        import torch
        self.vs = vs
        self.host_g = [g.cpu().pin_memory() for g in vs.grads]
        self.host_w = torch.empty(vs.n, dtype=torch.float32).pin_memory()
        self.copy_streams = [torch.cuda.Stream(device) for _ in range(4)]
        self.out_stream = torch.cuda.Stream(device)
        # Kernel completions are recorded on a stream of their own, so a
        # bucket's next copy-in does not queue behind another bucket's
        # copy-out.
        self.event_stream = torch.cuda.Stream(device)
        o = vs.offs
        self.spans = [(int(o[min(b)]), int(o[max(b) + 1]), vs.reducer.marks(b)) for b in vs.buckets]
        self.kernel_done = [torch.cuda.Event() for _ in self.spans]
        self.out_done = [torch.cuda.Event() for _ in self.spans]

    def start(self, stream):
        """Order the copy streams after ``stream`` (the start of a region)."""
        for cs in self.copy_streams + [self.out_stream, self.event_stream]:
            cs.wait_stream(stream)

    def step(self, stream):
        import torch
        vs, red = self.vs, self.vs.reducer
        k = 0
        for b, (lo, hi, ts) in enumerate(self.spans):
            used = []
            for r in range(P_VIT):
                cs = self.copy_streams[k % len(self.copy_streams)]
                k += 1
                if cs not in used:
                    used.append(cs)
                    cs.wait_event(self.kernel_done[b])
                with torch.cuda.stream(cs):
                    vs.grads[r][lo:hi].copy_(self.host_g[r][lo:hi], non_blocking=True)
            # The bucket's replicas arrive on several copy streams: join them
            # into one, and mark the bucket's tensors on it.
            for cs in used[1:]:
                used[0].wait_stream(cs)
            used[0].wait_event(self.out_done[b])
            red.mark_ready_many(ts, used[0])
            red.wait_bucket(b, self.event_stream)
            self.kernel_done[b].record(self.event_stream)
            red.wait_bucket(b, self.out_stream)
            with torch.cuda.stream(self.out_stream):
                self.host_w[lo:hi].copy_(vs.w[lo:hi], non_blocking=True)
            self.out_done[b].record(self.out_stream)
        red.finalize(stream)

    def finish(self, stream):
        """Order ``stream`` after every copy issued so far (the drain of a
        region)."""
        for cs in self.copy_streams + [self.out_stream, self.event_stream]:
            stream.wait_stream(cs)

    def copies_only(self, stream):
        """The step's host transfers alone, on the same streams and in the
        same pieces: every bucket's replicas in, its weights out, no kernel.
        Their time is the host link's bound on the end-to-end step.  As in
        ``step``, a bucket's copy-in waits for nothing but its own stream
        and a region ends with ``finish``."""
        import torch
        vs = self.vs
        k = 0
        for lo, hi, _ in self.spans:
            for r in range(P_VIT):
                cs = self.copy_streams[k % len(self.copy_streams)]
                k += 1
                with torch.cuda.stream(cs):
                    vs.grads[r][lo:hi].copy_(self.host_g[r][lo:hi], non_blocking=True)
            with torch.cuda.stream(self.out_stream):
                self.host_w[lo:hi].copy_(vs.w[lo:hi], non_blocking=True)


E2E_REGION_STEPS = 10   # steps per e2e region (fewer when --steps is smaller)
E2E_REGIONS = 31        # regions of each kind, interleaved


def time_e2e(args, device, stream):
    """The ViT step end to end from pinned host buffers (E2EStep), and the
    same transfers without the kernels (the host link's bound), measured
    alike: after 3 warm-up steps, 31 regions of min(K, 10) steps each, every
    region under one event pair with the same fill (``start``) and drain
    (``finish``), interleaved so that both meet the same traffic on the
    shared host; each figure is the median region.  Other jobs' transfers
    on the shared host link come in bursts that slow every region they
    overlap; short regions keep the share of regions they touch, and so the
    median, low."""
    import torch
    import gradient_all_reduce_gb300 as gar
    comm = gar.ar_init(P_VIT, device.index, gar.AR_MEAN)
    vs = None
    try:
        vs = VitStep(comm, device)
        e2e = E2EStep(vs, device)
        steps = max(3, min(args.steps, E2E_REGION_STEPS))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)

        def region(fn):
            t0.record(stream)
            e2e.start(stream)
            for _ in range(steps):
                fn(stream)
            e2e.finish(stream)
            t1.record(stream)
            torch.cuda.synchronize(device)
            return t0.elapsed_time(t1) / 1e3 / steps

        full, link = [], []
        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e.step(stream)
                e2e.copies_only(stream)
            e2e.finish(stream)
            torch.cuda.synchronize(device)
            for _ in range(E2E_REGIONS):
                full.append(region(e2e.step))
                link.append(region(e2e.copies_only))
        el, ln = statistics.median(full), statistics.median(link)
        value = vs.step_bytes / el / 1e9
        bound = vs.step_bytes / ln / 1e9
        # Other jobs' traffic on the shared host link only ever slows a
        # region down: the fastest region of each kind is the least disturbed.
        best, best_link = min(full), min(link)
        return {"value": value, "unit": "GB/s",
                "h2d_bytes_per_step": 2 * vs.n * P_VIT, "d2h_bytes_per_step": 4 * vs.n,
                "steps": steps, "ms_per_step": el * 1e3,
                "ms_per_step_regions": [round(x * 1e3, 3) for x in full],
                "link_only_ms_per_step": ln * 1e3,
                "link_only_ms_per_step_regions": [round(x * 1e3, 3) for x in link],
                "link_bound_GBps": bound,
                "frac_of_link_bound": value / bound,
                "best_ms_per_step": best * 1e3, "best_link_only_ms_per_step": best_link * 1e3,
                "frac_of_link_bound_best": best_link / best,
                "statistic": (f"median of {E2E_REGIONS} regions of `steps` steps for both the step and "
                              "the link-only transfers, each region with the same fill and drain, "
                              "the two kinds interleaved; *_best: the fastest region of each kind"),
                "path": ("ar_reducer_* with per-bucket H2D on 4 copy streams and per-bucket D2H "
                         "of the updated weights after ar_reducer_wait_bucket; consecutive steps "
                         "ordered per bucket, not per step")}
    finally:
        if vs is not None:
            vs.close()
        gar.ar_destroy(comm)


def flush_l2(buf):
    """Evict L2 before a timed call: write one 256 MiB buffer (twice the L2),
    then read a second one, which writes the first one's dirty lines back and
    leaves only clean lines behind.  The timed call then reads its inputs
    from HBM and pays for no write-back of the flush (the cold, clean state
    that ncu's cache control also gives)."""
    buf[0].add_(1)
    buf[1].sum()


def time_sweep(device, stream):
    """Flat all-reduce (Mean, in place) GB/s for P = 2, 4, 8 at 64 MiB,
    256 MiB and 1 GiB per replica, fp32 and bf16; reduce-scatter,
    all-gather and broadcast at 256 MiB per replica, P = 4 and 8; and the
    latency of small all-reduces (4 KiB .. 1 MiB, P = 8, fp32) and of
    SyncBN statistics, each also as one of 20 dependent calls replayed from
    one CUDA graph (chained_us).  L2 is
    flushed between repetitions (flush_l2: a 256 MiB write, then a 256 MiB
    read)."""
    import torch
    import gradient_all_reduce_gb300 as gar
    from workloads import gpu as wgpu
    flush = [torch.zeros(64 << 20, dtype=torch.float32, device=device) for _ in range(2)]
    out = {"all_reduce": [], "reduce_scatter": [], "all_gather": [], "broadcast": [],
           "small_all_reduce_us": []}

    def timed(fn, reps, flush_between=True):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                if flush_between:
                    flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                if i >= 3:
                    ts.append((e0, e1))
            torch.cuda.synchronize(device)
        return statistics.median(a.elapsed_time(b) / 1e3 for a, b in ts)

    def chained(call, k=20):
        """Per-call time of k calls captured in one CUDA graph, each kernel
        chained to the one before by programmatic dependent launch: the
        cost of one more dependent call in a sequence, launch overlapped
        (the *_us rows beside it time a call alone, its launch included)."""
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        call(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cur = torch.cuda.current_stream()
            for _ in range(k):
                call(cur)
        with torch.cuda.stream(stream):
            graph.replay()
            torch.cuda.synchronize(device)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            for i in range(5):
                ev[i].record(stream)
                graph.replay()
            ev[5].record(stream)
            torch.cuda.synchronize(device)
        del graph
        return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(5)) / 1e3 / k

    for P in (2, 4, 8):
        comm = gar.ar_init(P, device.index, gar.AR_MEAN)
        try:
            for dt, s in ((gar.AR_F32, 4), (gar.AR_BF16, 2)):
                tdt = torch.float32 if s == 4 else torch.bfloat16
                for mib in (64, 256, 1024):
                    n = (mib << 20) // s
                    xs = [torch.empty(n, dtype=tdt, device=device) for _ in range(P)]
                    for r, x in enumerate(xs):
                        wgpu.fill(x, "uniform", r)
                    t = timed(lambda: gar.ar_all_reduce(comm, xs, xs, n, dt, gar.AR_MEAN, stream),
                              10)
                    out["all_reduce"].append({"P": P, "dtype": "f32" if s == 4 else "bf16",
                                              "MiB_per_replica": mib, "us": t * 1e6,
                                              "GBps": 2 * P * n * s / t / 1e9})
                    del xs
            if P in (4, 8):
                n = (256 << 20) // 4
                shard = n // P
                xs = [torch.empty(n, dtype=torch.float32, device=device) for _ in range(P)]
                for r, x in enumerate(xs):
                    wgpu.fill(x, "uniform", r)
                rs = [torch.empty(shard, dtype=torch.float32, device=device) for _ in range(P)]
                t = timed(lambda: gar.ar_reduce_scatter(comm, xs, rs, n, gar.AR_F32, gar.AR_SUM,
                                                        stream), 10)
                out["reduce_scatter"].append({"P": P, "MiB_per_replica": 256, "us": t * 1e6,
                                              "GBps": (P + 1) * shard * P * 4 / t / 1e9})
                ins = [x[r * shard:(r + 1) * shard] for r, x in enumerate(xs)]
                t = timed(lambda: gar.ar_all_gather(comm, ins, xs, n, gar.AR_F32, stream), 10)
                out["all_gather"].append({"P": P, "MiB_per_replica": 256, "us": t * 1e6,
                                          "GBps": P * n * 4 / t / 1e9})
                t = timed(lambda: gar.ar_broadcast(comm, xs, n, gar.AR_F32, 0, stream), 10)
                out["broadcast"].append({"P": P, "MiB_per_replica": 256, "us": t * 1e6,
                                         "GBps": P * n * 4 / t / 1e9})
                del xs, rs, ins
            if P == 8:
                for kib in (4, 64, 1024):
                    n = (kib << 10) // 4
                    xs = [torch.empty(n, dtype=torch.float32, device=device) for _ in range(P)]
                    t_api = timed(lambda: gar.ar_all_reduce(comm, xs, xs, n, gar.AR_F32,
                                                            gar.AR_MEAN, stream),
                                  200, flush_between=False)
                    call = gar.PreparedCall("ar_all_reduce", comm, xs, xs, n, gar.AR_F32,
                                            gar.AR_MEAN)
                    t_prep = timed(lambda: call(stream), 200, flush_between=False)
                    side = torch.cuda.Stream(device)
                    side.wait_stream(stream)
                    call(side)
                    torch.cuda.synchronize(device)
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph):
                        call(torch.cuda.current_stream())
                    t_graph = timed(graph.replay, 200, flush_between=False)
                    del graph
                    t_chain = chained(call)
                    out["small_all_reduce_us"].append({"P": P, "KiB_per_replica": kib,
                                                       "api_us": t_api * 1e6,
                                                       "prepared_us": t_prep * 1e6,
                                                       "graph_us": t_graph * 1e6,
                                                       "chained_us": t_chain * 1e6})
                    del xs
        finally:
            gar.ar_destroy(comm)
    # No_sync accumulation on one ViT-sized bucket (25 MiB of bf16 per
    # replica, P = 8): a micro-batch before the last (acc += g / M) and the
    # last one fused with the all-reduce and the SGD step.
    comm = gar.ar_init(8, device.index, gar.AR_MEAN)
    try:
        P, n = 8, (25 << 20) // 2
        g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
        for r, x in enumerate(g):
            wgpu.fill(x, "normal", 100 + r, std=1e-3)
        acc = [torch.zeros(n, dtype=torch.float32, device=device) for _ in range(P)]
        w = torch.zeros(n, dtype=torch.float32, device=device)
        v = torch.zeros(n, dtype=torch.float32, device=device)
        ts, accs = [[x for x in g]], [[a for a in acc]]
        t_first = timed(lambda: gar.ar_bucket_accumulate(comm, ts, [n], gar.AR_BF16, accs, 0.25,
                                                         True, stream), 10)
        t_mid = timed(lambda: gar.ar_bucket_accumulate(comm, ts, [n], gar.AR_BF16, accs, 0.25,
                                                       False, stream), 10)
        t_last = timed(lambda: gar.ar_bucket_all_reduce_accumulated(
            comm, ts, [n], gar.AR_BF16, accs, 0.25, False, gar.AR_MEAN,
            sgd=(0.1, 0.9, [w], [v], 1), stream=stream), 10)
        out["accumulate_bucket_25MiB_P8_bf16"] = {
            "first_us": t_first * 1e6, "first_GBps": 6 * P * n / t_first / 1e9,
            "next_us": t_mid * 1e6, "next_GBps": 10 * P * n / t_mid / 1e9,
            "last_fused_sgd_us": t_last * 1e6,
            "last_fused_sgd_GBps": (8 * P * n + 16 * n) / t_last / 1e9}
        del g, acc, w, v
    finally:
        gar.ar_destroy(comm)
    # ZeRO-1 sharded step on the ViT-B/16 gradient set as one flat unit
    # (P = 8, bf16): reduce-scatter + owner's SGD + all-gather in one pass.
    # The unit is padded (86,567,656 -> 86,567,680) so each rank's shard is a
    # whole number of 16-byte vectors.
    comm = gar.ar_init(8, device.index, gar.AR_MEAN)
    try:
        P = 8
        n = -(-86_567_656 // (P * 8)) * (P * 8)
        sh = n // P
        g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
        for r, x in enumerate(g):
            wgpu.fill(x, "normal", 100 + r, std=1e-3)
        params = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
        ws = [torch.zeros(sh, dtype=torch.float32, device=device) for _ in range(P)]
        vs = [torch.zeros(sh, dtype=torch.float32, device=device) for _ in range(P)]
        t = timed(lambda: gar.ar_sharded_sgd_step(comm, g, params, ws, vs, n, gar.AR_BF16, 0.1,
                                                  0.9, gar.AR_MEAN, stream), 10, flush_between=False)
        out["zero1_sharded_step_vit_b16_P8_bf16"] = {
            "us": t * 1e6, "GBps": (4 * P * n + 16 * n) / t / 1e9}
        del g, params, ws, vs
    finally:
        gar.ar_destroy(comm)
    # Synchronized batch-norm statistics (P = 8): latency of one call through
    # the API, and of the same call replayed from a CUDA graph.
    comm = gar.ar_init(8, device.index, gar.AR_SUM)
    try:
        res = []
        for C in (64, 512, 2048):
            P = 8
            sums = [torch.rand(C, device=device) for _ in range(P)]
            sq = [torch.rand(C, device=device) + 1 for _ in range(P)]
            means = [torch.empty(C, device=device) for _ in range(P)]
            invs = [torch.empty(C, device=device) for _ in range(P)]

            def call(s=None):
                gar.ar_syncbn_stats(comm, sums, sq, [1000] * P, means, invs, C, 1e-5,
                                    stream if s is None else s)
            t_api = timed(call, 200, flush_between=False)
            prep = gar.PreparedCall("ar_syncbn_stats", comm, sums, sq, [1000] * P, means, invs,
                                    C, 1e-5)
            t_prep = timed(lambda: prep(stream), 200, flush_between=False)
            side = torch.cuda.Stream(device)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                call(side)
            torch.cuda.synchronize(device)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                call(torch.cuda.current_stream())
            t_graph = timed(graph.replay, 200, flush_between=False)
            del graph
            t_chain = chained(prep)
            res.append({"P": P, "channels": C, "api_us": t_api * 1e6,
                        "prepared_us": t_prep * 1e6, "graph_us": t_graph * 1e6,
                        "chained_us": t_chain * 1e6})
        out["syncbn_stats_latency"] = res
    finally:
        gar.ar_destroy(comm)
    del flush
    torch.cuda.empty_cache()
    return out


# -------------------------------------------------------------- CPU oracle
# The oracle is plain, single-threaded code.  Its Mean + SGD step is
# elementwise, so the unchanged oracle function called from several host
# threads on disjoint contiguous element ranges computes exactly the bits
# of one call over all elements (ctypes releases the interpreter lock for
# the duration of each call).  Nothing here imports the CUDA library.

def host_cores() -> int:
    """Host CPUs this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def vit_numel() -> int:
    import workloads
    return sum(workloads.vit_b16_numels())


def oracle_inputs(elems: int, offset: int = 0, threads: int = 1):
    """Host inputs of ``elems`` contiguous gradient elements of the ViT step
    starting at ``offset``: every replica's bf16 gradients, the fp32 master
    weights and zero momentum.  Drawn chunk by chunk over ``threads``."""
    from concurrent.futures import ThreadPoolExecutor
    import workloads
    grads = [np.empty(elems, np.uint16) for _ in range(P_VIT)]
    w = np.empty(elems, np.float32)
    v = np.zeros(elems, np.float32)
    chunk = 1 << 22

    def fill(lo):
        hi = min(elems, lo + chunk)
        for r in range(P_VIT):
            grads[r][lo:hi] = workloads.replica_values(
                "normal", "bf16", workloads.VIT_GRAD_SEED + r, hi - lo,
                std=workloads.VIT_GRAD_STD, start=offset + lo)
        w[lo:hi] = workloads.normal_f32(workloads.VIT_MASTER_SEED, hi - lo,
                                        std=workloads.VIT_MASTER_STD, start=offset + lo)

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(fill, range(0, elems, chunk)))
    return grads, w, v


def oracle_step(inputs, threads: int = 1, pool=None) -> None:
    """One Mean + SGD step (momentum 0.9, lr 0.1, write-back) of the oracle
    over all of ``inputs``, in place: the oracle's bucket all-reduce called
    once per thread on ``threads`` disjoint contiguous element ranges."""
    import oracle
    grads, w, v = inputs
    n = w.size
    if threads <= 1 or pool is None:
        oracle.bucket_all_reduce([grads], op=oracle.MEAN, sgd=(0.1, 0.9, [w], [v], 1))
        return
    cuts = [n * k // threads for k in range(threads + 1)]

    def run(k):
        lo, hi = cuts[k], cuts[k + 1]
        if hi > lo:
            oracle.bucket_all_reduce([[g[lo:hi] for g in grads]], op=oracle.MEAN,
                                     sgd=(0.1, 0.9, [w[lo:hi]], [v[lo:hi]], 1))

    list(pool.map(run, range(threads)))


def oracle_rate(inputs, threads: int, min_seconds: float, min_reps: int = 1):
    """Repeat oracle_step until min_seconds (and min_reps) have passed;
    returns (GB/s of algorithmic bytes, repetitions, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.lib()
    n = inputs[1].size
    with ThreadPoolExecutor(threads) as pool:
        oracle_step(inputs, threads, pool)            # first touch of every page
        reps, spent = 0, 0.0
        while spent < min_seconds or reps < min_reps:
            t0 = time.perf_counter()
            oracle_step(inputs, threads, pool)
            spent += time.perf_counter() - t0
            reps += 1
    return vit_bytes(n) * reps / spent / 1e9, reps, spent


def cpu_baseline_full(min_seconds: float = 3.0):
    """The oracle on the whole ViT step (every one of the 86,567,656
    gradient elements of all 8 replicas), on all host cores and on one."""
    import oracle
    oracle.build()
    cores = host_cores()
    n = vit_numel()
    inputs = oracle_inputs(n, threads=cores)
    rate_all, reps_all, spent_all = oracle_rate(inputs, cores, min_seconds, min_reps=3)
    rate_one, reps_one, spent_one = oracle_rate(inputs, 1, min_seconds, min_reps=1)
    what = (f"the oracle's Mean + SGD step (write-back) over all {n:,} gradient elements of "
            f"all {P_VIT} replicas")
    return {"value": rate_all, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": (f"{reps_all} runs of {what}, the unchanged oracle function called from "
                       f"{cores} host threads on disjoint contiguous element ranges, "
                       f"{spent_all:.1f} s"),
            "single_thread": {"value": rate_one, "unit": "GB/s", "cores": 1,
                              "sample": f"{reps_one} runs of {what} in one call, {spent_one:.1f} s"}}


def run_reference(args):
    """The CPU oracle, timed on all host cores: each step is the oracle's
    Mean + SGD over the whole ViT step when K + W such steps fit a bounded
    budget, else over one contiguous slice of it; rank 0 only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = host_cores()
    n_total = vit_numel()
    probe = oracle_inputs(1 << 22, threads=cores)
    rate, _, _ = oracle_rate(probe, cores, 0.5)
    del probe
    per_step_s = args.ref_budget / max(1, args.steps + args.warmup)
    elems = int(max(1 << 16, min(n_total, rate * 1e9 * per_step_s / vit_bytes(1))))
    inputs = oracle_inputs(elems, threads=cores)
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(cores) as pool:
        for _ in range(args.warmup):
            oracle_step(inputs, cores, pool)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_step(inputs, cores, pool)
        el = time.perf_counter() - t0
    value = vit_bytes(elems) * args.steps / el / 1e9
    part = ("all" if elems == n_total else f"the first {elems:,} of the")
    sample = (f"each step: the oracle's Mean + SGD step (write-back) on {part} {n_total:,} "
              f"gradient elements of all {P_VIT} replicas, the unchanged oracle function called "
              f"from {cores} host threads on disjoint contiguous element ranges")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": vit_config(args.gpus),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- overlap

def vit_b16_module(device, dtype):
    """ViT-B/16 as the "Distributed Training" page builds it (patch 16,
    width 768, 12 pre-norm encoder blocks, MLP 3072, 1000 classes), with
    random initial weights."""
    import torch
    import torch.nn as nn
    import workloads

    class ViT(nn.Module):
        def __init__(self):
            super().__init__()
            D = workloads.VIT_D
            self.patch = nn.Conv2d(3, D, workloads.VIT_PATCH, stride=workloads.VIT_PATCH)
            self.cls = nn.Parameter(torch.zeros(1, 1, D))
            self.pos = nn.Parameter(torch.randn(1, workloads.VIT_TOKENS, D) * 0.02)
            self.blocks = nn.ModuleList(
                nn.TransformerEncoderLayer(D, 12, workloads.VIT_MLP, dropout=0.0, norm_first=True,
                                           batch_first=True) for _ in range(workloads.VIT_LAYERS))
            self.norm, self.head = nn.LayerNorm(D), nn.Linear(D, workloads.VIT_CLASSES)

        def forward(self, x):
            h = self.patch(x).flatten(2).transpose(1, 2)
            h = torch.cat([self.cls.expand(h.shape[0], -1, -1), h], dim=1) + self.pos
            for blk in self.blocks:
                h = blk(h)
            return self.head(self.norm(h[:, 0]))

    torch.manual_seed(0)
    return ViT().to(device=device, dtype=dtype)


def run_overlap(args):
    """DDP's point: hide the all-reduce behind the backward pass.  Rank 0's
    forward + backward of ViT-B/16 (bf16) runs on the GPU while the
    reducer launches each bucket (P = 8 replicas, Mean + fused SGD) from the
    autograd hooks as its gradients become final; ranks 1..7's gradients
    are synthetic.  Reports forward+backward alone, the gradient step
    alone, and both overlapped."""
    import torch
    import gradient_all_reduce_gb300 as gar
    from gradient_all_reduce_gb300.ddp import ReplicaDDP
    from workloads import gpu as wgpu
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    model = vit_b16_module(device, torch.bfloat16)
    comm = gar.ar_init(P_VIT, 0, gar.AR_MEAN)
    ddp = ReplicaDDP(comm, model, P_VIT, CAP, gar.AR_MEAN, sgd=(0.1, 0.9))
    try:
        for r in range(1, P_VIT):
            wgpu.fill(ddp.flat[r], "normal", 100 + r, std=1e-3)
        g = torch.Generator(device=device).manual_seed(0)
        x = torch.randn(args.batch, 3, 224, 224, device=device, dtype=torch.bfloat16, generator=g)
        y = torch.randint(0, 1000, (args.batch,), device=device, generator=g)
        reverse = list(range(len(ddp.params) - 1, -1, -1))

        def fwd_bwd(hooks):
            ddp.hooks_enabled = hooks
            ddp.flat[0].zero_()
            torch.nn.functional.cross_entropy(model(x), y).backward()
            if hooks:
                ddp.finish()

        def sync_only():
            s = torch.cuda.current_stream()     # the capture stream while graphing
            ddp.reducer.mark_ready_many(reverse, s)
            ddp.finish(s)

        def timed(fn, reps):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        def graphed(fn):
            """fn captured in a CUDA graph (after warm-up on a side stream):
            replays carry no host overhead, so only GPU-side overlap shows."""
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(3):
                    fn()
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fn()
            return graph.replay

        reps = max(5, min(args.steps, 50))
        eager = {"fwd_bwd_ms": timed(lambda: fwd_bwd(False), reps),
                 "grad_step_ms": timed(sync_only, reps),
                 "overlapped_ms": timed(lambda: fwd_bwd(True), reps),
                 "sequential_ms": timed(lambda: (fwd_bwd(False), sync_only()), reps)}
        g_fb, g_sync = graphed(lambda: fwd_bwd(False)), graphed(sync_only)
        g_ov = graphed(lambda: fwd_bwd(True))
        graphs = {"fwd_bwd_ms": timed(g_fb, reps), "grad_step_ms": timed(g_sync, reps),
                  "overlapped_ms": timed(g_ov, reps),
                  "sequential_ms": timed(lambda: (g_fb(), g_sync()), reps)}
        for d in (eager, graphs):
            d["hidden_fraction"] = (d["sequential_ms"] - d["overlapped_ms"]) / d["grad_step_ms"]
            d["speedup_vs_sequential"] = d["sequential_ms"] / d["overlapped_ms"]
        if gar.ar_get_async_error(comm) != gar.AR_OK:
            raise RuntimeError("device status")
        print(json.dumps({
            "mode": "overlap", "model": "ViT-B/16 (bf16, random init)", "batch": args.batch,
            "P": P_VIT, "buckets": len(set(ddp.reducer.bucket_of())), "reps": reps,
            "cuda_graphs": graphs, "eager": eager}), flush=True)
    finally:
        ddp.close()
        gar.ar_destroy(comm)


# ------------------------------------------------------------ full sweep

SWEEP_KIB = [4 << (2 * k) for k in range(10)]          # 4 KiB .. 1 GiB per replica
L2_BYTES = 129 * 10 ** 6                               # GB300 L2


def run_full_sweep(args):
    """All-reduce GB/s and fraction of the HBM roofline against message size:
    per replica 4 KiB * 4^k (k = 0..9), P = 2, 4, 8, fp32 and bf16, Sum and
    Mean, in place; and broadcast from rank 0 at the same sizes.  Each row
    is the median of event-timed calls on one stream, each preceded by a
    256 MiB write and a 256 MiB read that leave L2 clean and cold (flush_l2);
    5 warm-up calls, 20 timed (200 below 1 MiB).  Rows below 1 MiB also
    give the latency of back-to-back calls through the API and as a
    replayed CUDA graph (no flush: the launch cost is what they measure).
    Rows whose P replicas hold at least twice the L2 also give the rate of
    20 calls back to back without a flush, where each call pays for the
    previous call's writes still dirty in L2 (the steady state; a call
    after the flush does not pay for its own).
    Sum rows repeat on the same buffers (values may overflow to inf; the
    kernels' time does not depend on values).  One JSON line; rank 0 of a
    single process only."""
    import torch
    import gradient_all_reduce_gb300 as gar
    from workloads import gpu as wgpu
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peak, peak_kind = measured_peak()
    flush = [torch.zeros(64 << 20, dtype=torch.float32, device=device) for _ in range(2)]

    def median_time(fn, reps, flush_between):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(reps + 5):
                if flush_between:
                    flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                if i >= 5:
                    ts.append((e0, e1))
            torch.cuda.synchronize(device)
        return statistics.median(a.elapsed_time(b) / 1e3 for a, b in ts)

    def back_to_back(call, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                call(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                call(stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) / 1e3 / reps

    def graph_of(fn):
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn(torch.cuda.current_stream())
        return graph

    rows = []
    t_start = time.perf_counter()
    with ClockSampler(0) as clocks:
        # The floor of one launch, measured the same ways: a one-CTA torch
        # kernel on 4 KiB (event-timed after the flush, back to back, and as
        # a replayed one-node CUDA graph).
        tiny = torch.zeros(1024, dtype=torch.float32, device=device)
        g_tiny = graph_of(lambda s: tiny.add_(1))
        floor = {"what": "torch add_ on 4 KiB (one small kernel), timed like the rows",
                 "us": 1e6 * median_time(lambda: tiny.add_(1), 200, True),
                 "api_us": 1e6 * median_time(lambda: tiny.add_(1), 200, False),
                 "graph_us": 1e6 * median_time(g_tiny.replay, 200, False)}
        del g_tiny
        for P in (2, 4, 8):
            comm = gar.ar_init(P, 0, gar.AR_MEAN)
            try:
                for dt, es, tdt, name in ((gar.AR_F32, 4, torch.float32, "f32"),
                                          (gar.AR_BF16, 2, torch.bfloat16, "bf16")):
                    nmax = (SWEEP_KIB[-1] << 10) // es
                    bufs = [torch.empty(nmax, dtype=tdt, device=device) for _ in range(P)]
                    for kib in SWEEP_KIB:
                        n = (kib << 10) // es
                        small = kib < 1024
                        reps = 200 if small else 20
                        xs = [b[:n] for b in bufs]
                        for op, opname in ((gar.AR_SUM, "sum"), (gar.AR_MEAN, "mean"),
                                           (None, "broadcast")):
                            for r, x in enumerate(xs):
                                wgpu.fill(x, "uniform", r)
                            if op is None:
                                call = gar.PreparedCall("ar_broadcast", comm, xs, n, dt, 0)
                                nbytes = P * n * es
                            else:
                                call = gar.PreparedCall("ar_all_reduce", comm, xs, xs, n, dt, op)
                                nbytes = 2 * P * n * es
                            if op is None:
                                t = median_time(lambda: gar.ar_broadcast(comm, xs, n, dt, 0, stream),
                                                reps, True)
                            else:
                                t = median_time(lambda: gar.ar_all_reduce(comm, xs, xs, n, dt, op,
                                                                          stream), reps, True)
                            row = {"op": opname, "P": P, "dtype": name, "KiB_per_replica": kib,
                                   "bytes": nbytes, "us": t * 1e6, "GBps": nbytes / t / 1e9,
                                   "frac": nbytes / t / 1e9 / peak}
                            if P * n * es >= 2 * L2_BYTES:
                                # Steady state of repeated calls: each call also
                                # writes back the previous one's dirty lines.
                                tb = back_to_back(call, 20)
                                row["b2b_GBps"] = nbytes / tb / 1e9
                                row["b2b_frac"] = nbytes / tb / 1e9 / peak
                            if small:
                                row["api_us"] = 1e6 * median_time(
                                    lambda: call(stream), reps, False)
                                g = graph_of(call)
                                row["graph_us"] = 1e6 * median_time(g.replay, reps, False)
                                del g
                            rows.append(row)
                    del bufs, xs
                    torch.cuda.empty_cache()
                if gar.ar_get_async_error(comm) != gar.AR_OK:
                    raise RuntimeError("device status")
            finally:
                gar.ar_destroy(comm)
    # The oracle beside it: its in-place Mean all-reduce on the host, as it
    # stands (one thread), on 4 MiB per replica of the same uniform inputs,
    # repeated for at least half a second per cell.
    import oracle
    import workloads
    oracle.build()
    cpu_rows = []
    for P in (2, 4, 8):
        for name, es in (("f32", 4), ("bf16", 2)):
            n = (4 << 20) // es
            xs = [workloads.replica_values("uniform", name, r, n) for r in range(P)]
            reps, spent = 0, 0.0
            while spent < 0.5 or reps == 0:
                t0 = time.perf_counter()
                oracle.all_reduce(xs, recv=xs, op=oracle.MEAN)
                spent += time.perf_counter() - t0
                reps += 1
            cpu_rows.append({"op": "mean", "P": P, "dtype": name, "KiB_per_replica": 4096,
                             "GBps": 2 * P * n * es * reps / spent / 1e9, "reps": reps,
                             "cores": 1})
    print(json.dumps({
        "mode": "sweep", "metric": METRIC, "peak_GBps": peak, "peak_kind": peak_kind,
        "bytes": "all-reduce 2*P*N*s, broadcast P*N*s (every replica read and written once)",
        "timing": ("median of event-timed calls after a 256 MiB write and a 256 MiB read "
                   "(L2 cold and clean); 5 warm-up, "
                   "20 timed (200 below 1 MiB); api_us / graph_us: back-to-back calls, no flush"),
        "seconds": time.perf_counter() - t_start, "clocks": clocks.summary(),
        "launch_floor": floor, "rows": rows,
        "cpu_oracle": {"kind": "oracle", "cores": 1, "host_cpus": os.cpu_count(),
                       "rows": cpu_rows}}), flush=True)


# ------------------------------------------------------------------ cases

def case_cpu_baseline(case, P, dtype_name, op_name, min_seconds=1.0):
    """The oracle beside a --case line: the oracle as it stands (one
    thread) on a bounded sample of the case's workload, 2**20 elements per
    replica (the 2048 channels for syncbn), the same seeded inputs, repeated
    for at least min_seconds; GB/s by the case's algorithmic-bytes formula."""
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    op = oracle.SUM if op_name == "sum" else oracle.MEAN
    n = (1 << 20) // (8 * P) * (8 * P)
    if case in ("ar", "rs", "ag", "bc"):
        es = 4 if dtype_name == "f32" else 2
        xs = [workloads.replica_values("uniform", dtype_name, r, n) for r in range(P)]
        sh = n // P
        if case == "ar":
            fn, nbytes = (lambda: oracle.all_reduce(xs, recv=xs, op=op)), 2 * P * n * es
        elif case == "rs":
            out = [np.empty(sh, xs[0].dtype) for _ in range(P)]
            fn, nbytes = (lambda: oracle.reduce_scatter(xs, recv=out, op=op)), (P + 1) * n * es
        elif case == "ag":
            shards = [x[r * sh:(r + 1) * sh].copy() for r, x in enumerate(xs)]
            fn, nbytes = (lambda: oracle.all_gather(shards, recv=xs)), P * n * es
        else:
            fn, nbytes = (lambda: oracle.broadcast(xs, 0)), P * n * es
        sample = f"{n} {dtype_name} elements per replica"
    elif case == "zero1":
        g = [workloads.replica_values("normal", "bf16", 100 + r, n, std=1e-3) for r in range(P)]
        params = [np.zeros(n, np.uint16) for _ in range(P)]
        ws = [np.zeros(n // P, np.float32) for _ in range(P)]
        vs = [np.zeros(n // P, np.float32) for _ in range(P)]
        fn = lambda: oracle.sharded_sgd_step(g, params, ws, vs, 0.1, 0.9, oracle.MEAN)
        nbytes, sample = 4 * P * n + 16 * n, f"a flat unit of {n} bf16 elements"
    elif case == "sgd":
        g = [[workloads.replica_values("normal", "bf16", 100 + r, n, std=1e-3) for r in range(P)]]
        w, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
        fn = lambda: oracle.bucket_all_reduce(g, op=oracle.MEAN, sgd=(0.1, 0.9, [w], [v], 1))
        nbytes, sample = 4 * P * n + 16 * n, f"one bucket of {n} bf16 elements per replica"
    elif case in ("accfirst", "acc", "acclast"):
        g = [[workloads.replica_values("normal", "bf16", 100 + r, n, std=1e-3) for r in range(P)]]
        acc = [[np.zeros(n, np.float32) for _ in range(P)]]
        if case == "acclast":
            w, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
            fn = lambda: oracle.bucket_all_reduce_accumulated(g, acc, 0.25, False, oracle.MEAN,
                                                              sgd=(0.1, 0.9, [w], [v], 1))
            nbytes = 8 * P * n + 16 * n
        else:
            first = case == "accfirst"
            fn = lambda: oracle.bucket_accumulate(g, acc, 0.25, first)
            nbytes = (6 if first else 10) * P * n
        sample = f"one bucket of {n} bf16 elements per replica"
    else:
        C = 2048
        sums = [workloads.uniform_f32(r, C) for r in range(P)]
        sq = [workloads.uniform_f32(100 + r, C) + np.float32(1) for r in range(P)]
        fn = lambda: oracle.syncbn_stats(sums, sq, [1000] * P, 1e-5)
        nbytes, sample = 4 * P * C * 4, f"{C} channels"
    reps, spent = 0, 0.0
    while spent < min_seconds or reps == 0:
        t0 = time.perf_counter()
        fn()
        spent += time.perf_counter() - t0
        reps += 1
    return {"value": nbytes * reps / spent / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{sample}, P={P}, {reps} calls in {spent:.2f} s, one thread"}


def run_case(args):
    """One collective alone and one JSON line: K calls back to back after W
    warm-up calls (us, GBps, frac), then the median of 20 calls each timed
    alone from a cold, clean L2 (us_cold, GBps_cold, frac_cold).  256 MiB
    per replica for ar / rs / ag / bc (P and the element type from
    --case-ranks and --case-dtype; P = 8, fp32 by default); one 25 MiB bf16
    bucket for sgd, accfirst, acc and acclast (P from --case-ranks); the ViT-B/16 gradient
    set (bf16, P = 8) for zero1.  Also the host's issue time per call in the
    back-to-back loop (host_us) and the K calls replayed from one CUDA graph
    (us_graph, GBps_graph, frac_graph)."""
    import torch
    import gradient_all_reduce_gb300 as gar
    from workloads import gpu as wgpu
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    if args.case == "tiny":   # the tiny all-reduce: P = 4, 2**20 fp32 per replica, Mean, in place
        args.case, args.case_ranks, args.case_mib = "ar", 4, 4
        args.case_dtype, args.case_op = "f32", "mean"
    flat = args.case in ("ar", "rs", "ag", "bc")
    P = args.case_ranks if flat or args.case.startswith("acc") or args.case == "sgd" else 8
    comm = gar.ar_init(P, 0, gar.AR_MEAN)
    try:
        if flat:
            es, tdt, dt = ((4, torch.float32, gar.AR_F32) if args.case_dtype == "f32"
                           else (2, torch.bfloat16, gar.AR_BF16))
            n = (args.case_mib << 20) // es // (8 * P) * (8 * P)  # whole 16-byte vectors per shard
            op_name = args.case_op or ("mean" if args.case == "ar" else "sum")
            op = gar.AR_SUM if op_name == "sum" else gar.AR_MEAN
            xs = [torch.empty(n, dtype=tdt, device=device) for _ in range(P)]
            for r, x in enumerate(xs):
                wgpu.fill(x, "uniform", r)
            sh = n // P
            rs = [torch.empty(sh, dtype=tdt, device=device) for _ in range(P)]
            ins = [x[r * sh:(r + 1) * sh] for r, x in enumerate(xs)]
            prep, nbytes = {
                "ar": (gar.PreparedCall("ar_all_reduce", comm, xs, xs, n, dt, op), 2 * P * n * es),
                "rs": (gar.PreparedCall("ar_reduce_scatter", comm, xs, rs, n, dt, op),
                       (P + 1) * n * es),
                "ag": (gar.PreparedCall("ar_all_gather", comm, ins, xs, n, dt), P * n * es),
                "bc": (gar.PreparedCall("ar_broadcast", comm, xs, n, dt, 0), P * n * es),
            }[args.case]
            call = prep
            what = f"P={P} {args.case_dtype} {args.case_mib} MiB per replica"
            if args.case in ("ar", "rs"):
                what += f", {op_name}"
        elif args.case == "zero1":
            n = -(-86_567_656 // (P * 8)) * (P * 8)
            g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
            for r, x in enumerate(g):
                wgpu.fill(x, "normal", 100 + r, std=1e-3)
            params = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
            ws = [torch.zeros(n // P, device=device) for _ in range(P)]
            vs = [torch.zeros(n // P, device=device) for _ in range(P)]
            call = gar.PreparedCall("ar_sharded_sgd_step", comm, g, params, ws, vs, n, gar.AR_BF16,
                                    gar.AR_MEAN, 0.1, 0.9)
            nbytes, what = 4 * P * n + 16 * n, "ViT-B/16 flat unit, P=8 bf16"
        elif args.case == "sgd":
            n = (25 << 20) // 2
            g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
            for r, x in enumerate(g):
                wgpu.fill(x, "normal", 100 + r, std=1e-3)
            w, v = torch.zeros(n, device=device), torch.zeros(n, device=device)
            call = gar.PreparedBucket(comm, [g], [n], gar.AR_BF16, gar.AR_MEAN,
                                      sgd=(0.1, 0.9, [w], [v], 1))
            nbytes = 4 * P * n + 16 * n
            what = f"one 25 MiB bf16 bucket, P={P}, Mean + SGD with write-back"
        elif args.case in ("accfirst", "acc"):
            first = args.case == "accfirst"
            n = (25 << 20) // 2
            g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
            for r, x in enumerate(g):
                wgpu.fill(x, "normal", 100 + r, std=1e-3)
            acc = [[torch.zeros(n, device=device) for _ in range(P)]]
            call = lambda s: gar.ar_bucket_accumulate(comm, [g], [n], gar.AR_BF16, acc, 0.25,
                                                      first, s)
            nbytes = (6 if first else 10) * P * n
            what = (f"one 25 MiB bf16 bucket, P={P}, "
                    + ("the first micro-batch" if first else "a micro-batch before the last"))
        elif args.case == "acclast":
            n = (25 << 20) // 2
            g = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
            for r, x in enumerate(g):
                wgpu.fill(x, "normal", 100 + r, std=1e-3)
            acc = [[torch.zeros(n, device=device) for _ in range(P)]]
            w, v = torch.zeros(n, device=device), torch.zeros(n, device=device)
            call = lambda s: gar.ar_bucket_all_reduce_accumulated(
                comm, [g], [n], gar.AR_BF16, acc, 0.25, False, gar.AR_MEAN,
                sgd=(0.1, 0.9, [w], [v], 1), stream=s)
            nbytes = 8 * P * n + 16 * n
            what = f"one 25 MiB bf16 bucket, P={P}, the last micro-batch with Mean + SGD"
        else:
            C = 2048
            sums = [torch.rand(C, device=device) for _ in range(P)]
            sq = [torch.rand(C, device=device) + 1 for _ in range(P)]
            mo = [torch.empty(C, device=device) for _ in range(P)]
            io = [torch.empty(C, device=device) for _ in range(P)]
            call = gar.PreparedCall("ar_syncbn_stats", comm, sums, sq, [1000] * P, mo, io, C, 1e-5)
            nbytes, what = 4 * P * C * 4, "P=8, 2048 channels"
        fn = lambda: call(stream)
        for _ in range(max(1, args.warmup)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h0 = time.perf_counter()
        for _ in range(args.steps):
            fn()
        host = (time.perf_counter() - h0) / args.steps
        e1.record(stream)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3 / args.steps
        # The same call alone from a cold, clean L2: median of event pairs.
        flush = [torch.empty(64 << 20, device=device) for _ in range(2)]
        pairs = []
        for _ in range(20):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            pairs.append((a, b))
        torch.cuda.synchronize()
        cold = statistics.median(a.elapsed_time(b) for a, b in pairs) / 1e3
        peak, _ = measured_peak()
        line = {"case": args.case, "workload": what, "us": t * 1e6, "GBps": nbytes / t / 1e9,
                "frac": nbytes / t / 1e9 / peak, "us_cold": cold * 1e6,
                "GBps_cold": nbytes / cold / 1e9, "frac_cold": nbytes / cold / 1e9 / peak,
                "host_us": host * 1e6}
        # The same calls replayed from one CUDA graph of K calls: no host
        # time between launches, consecutive kernels chained by
        # programmatic dependent launch (below ~40 MB per call the
        # operands stay in L2 from one call to the next).  Back to back
        # from the host, a call whose host issue time (host_us) is above
        # its device time leaves the GPU idle between calls; the graph
        # shows the device time alone.
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        call(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cur = torch.cuda.current_stream()
            for _ in range(args.steps):
                call(cur)
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        tg = e0.elapsed_time(e1) / 1e3 / args.steps
        line.update({"us_graph": tg * 1e6, "GBps_graph": nbytes / tg / 1e9,
                     "frac_graph": nbytes / tg / 1e9 / peak})
        del graph
        if not args.no_cpu:
            line["cpu_baseline"] = case_cpu_baseline(
                args.case, P, args.case_dtype if flat else "bf16",
                args.case_op or ("mean" if args.case == "ar" else "sum"))
        print(json.dumps(line), flush=True)
    finally:
        gar.ar_destroy(comm)


# -------------------------------------------------------------------- main

def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.overlap:
        run_overlap(args)
        return
    if args.case:
        run_case(args)
        return
    if args.sweep:
        run_full_sweep(args)
        return
    rank, world, local = dist_env()
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import gradient_all_reduce_gb300  # noqa: F401  (fails loudly without libgar.so)
    stream = torch.cuda.Stream(device)

    res = time_vit(args, device, stream, world)
    elapsed = max_over_ranks(res["elapsed"], world, device)
    total_bytes = res["step_bytes"] * args.steps * world
    value = total_bytes / elapsed / 1e9
    peak, peak_kind = measured_peak()
    achieved = res["step_bytes"] * args.steps / res["combined_s"] / 1e9
    per_bucket = res["launch_bytes"] / res["serial_s"] / 1e9
    achieved_events = res["launch_bytes"] / res["launch_s"] / 1e9
    traffic = committed_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": vit_config(world),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": ("k_reduce<BF16, P=8, SGD, CapLarge>: one launch over the 8 "
                                "buckets' 152 tensors (4.155 GB)"),
                     "note": ("the kernel the reducer launches in the headline region, issued "
                              "K times back to back on the timing stream under one CUDA-event "
                              "pair (second timed region), behind one untimed launch so that "
                              "the host's first issue is not counted: region time / K = "
                              "average launch duration"),
                     "achieved_per_bucket_launch": per_bucket,
                     "frac_per_bucket_launch": per_bucket / peak,
                     "per_bucket_note": ("the 8 bucket calls one after another on one stream "
                                         "(8 launches per step)"),
                     "achieved_per_launch_events": achieved_events,
                     "frac_per_launch_events": achieved_events / peak,
                     "traffic": traffic["dram_bytes_per_launch"] if traffic else None},
        "gpu_launches": res["launches"],
        "gpu_launches_note": ("kernel launches in the headline region, counted by the reducer "
                              "(ar_reducer_launches): the 8 buckets of a step complete in one "
                              "mark_ready_many call and go out as one combined launch"),
        "host_us_per_step": res["host_us_per_step"],
        "serialized_ms_per_step": res["serial_ms_per_step"],
        "combined_ms_per_step": res["combined_ms_per_step"],
        "clocks": res["clocks"],
    }
    if traffic:
        line["roofline"]["traffic_note"] = ("DRAM bytes read + written by one combined launch, "
                                            "from " + traffic["source"])
    if rank == 0 and not args.no_e2e:
        line["e2e"] = time_e2e(args, device, stream)
    if rank == 0 and not args.no_sweep:
        line["sweep"] = time_sweep(device, stream)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_full()
    barrier(world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
