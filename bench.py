"""Throughput of the collapse-safe CE forward+backward on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload pages|chunked|mid|linear|linear_peaked]

One step = ce_forward + ce_backward over one batch of the workload (default: the pages'
shape, T=16384 rows x V=128256 bf16 logits, mean over non-ignored rows, 10% of rows with
the target raised by 17..50 above the row max, 1% ignored).  Inputs are resident in HBM
before the timed region; the 4.2 GB logits are ~33x the 129 MB L2, so every pass streams
from HBM with no flush needed.  `value` is whole-job tokens/s (all ranks); `e2e` is the same
metric with the step's inputs copied from pinned host memory and the loss read back inside
the timed region.  `--impl reference` times the fp64 CPU oracle on a bounded row sample.

The default line also carries `linear`: the fused linear-CE (E [8192, 4096], W [128256, 4096]
bf16, linear_ce_fwd_bwd) timed the same way in its own region, with its tensor-core rate
against the measured bf16 peaks, the CUDA-event time of each of its GEMMs and its own clocks.

Under torchrun (--gpus N > 1) each rank runs an independent replica on its own batch
(rows are independent: no data-path collective); the timed region is bracketed by a
barrier and the max over ranks is taken.  Rank 0 prints one JSON line.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_DIR = os.path.join(ROOT, "profiles")


# ------------------------------------------------------------------------------- distributed plumbing

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------- peaks, clocks, profiles

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.devnull if False else f"/tmp/vce_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", f"-lms", str(self.period)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.out:
            self.out.close()

    def summary(self):
        path = f"/tmp/vce_clocks_{os.getpid()}.csv"
        if self.proc is None or not os.path.exists(path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in open(path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "active": parts[4], "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        os.remove(path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 200] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded),
                "power_w_max": max(r["power"] for r in rows)}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


RING_FILES = ["vocab_cross_entropy_gb300/csrc/ce_ring.cu", "vocab_cross_entropy_gb300/csrc/ce_stage.cuh",
              "vocab_cross_entropy_gb300/csrc/ce_fold.cuh", "vocab_cross_entropy_gb300/csrc/ce_slots.cuh",
              "vocab_cross_entropy_gb300/csrc/vce_device.cuh", "vocab_cross_entropy_gb300/csrc/vce_async.cuh"]


def captured_shape(w):
    """The committed DRAM captures are of T=16384, V=128256 bf16 logits, bf16 gradient, mean."""
    return (w.p.T, w.p.V, w.p.dtype, w.red, w.eps) == (16384, 128256, "bf16", "mean", 0.0)


def profiled_traffic(name, files):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(PROFILE_DIR, f"{name}.json")
    try:
        d = json.load(open(path))
    except Exception:
        return None
    if d.get("source_files", files) != files or d.get("source_hash") != kernel_source_hash(files):
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------- workloads

class CEWorkload:
    """The pages' shape (default) or the mid shape: ce_forward + ce_backward."""

    KERNEL_FILES = ["vocab_cross_entropy_gb300/csrc/ce_bwd.cu", "vocab_cross_entropy_gb300/csrc/ce_rows.cuh",
                    "vocab_cross_entropy_gb300/csrc/ce_segments.h", "vocab_cross_entropy_gb300/csrc/vce_device.cuh"]

    def __init__(self, problem, device, reduction="mean", label_smoothing=0.0):
        import vocab_cross_entropy_gb300 as vce
        self.vce = vce
        self.p = problem
        self.dev = device
        self.red = reduction
        self.eps = float(label_smoothing)
        T, V = problem.T, problem.V
        self.es = 2 if problem.dtype == "bf16" else 4
        tdt = torch.bfloat16 if problem.dtype == "bf16" else torch.float32
        self.host = torch.empty((T, V), dtype=torch.int16 if self.es == 2 else torch.float32, pin_memory=True)
        problem.full(out=self.host.numpy().view(problem.np_dtype))
        self.host_bf16 = self.host.view(tdt)          # the host logits in their storage dtype
        self.labels_host = torch.from_numpy(problem.labels).pin_memory()
        self.logits = self.host_bf16.to(device)
        self.labels = self.labels_host.to(device)
        self.loss_rows = torch.empty(T, dtype=torch.float32, device=device)
        self.loss_out = torch.empty(1, dtype=torch.float32, device=device)
        self.stats = torch.empty(T, 4, dtype=torch.float32, device=device)
        self.status = torch.empty(1, dtype=torch.int32, device=device)
        self.go = (torch.linspace(0.5, 1.5, T, dtype=torch.float32, device=device) if reduction == "none"
                   else torch.ones(1, dtype=torch.float32, device=device))
        self.grad = torch.empty((T, V), dtype=tdt, device=device)
        self.loss_host = torch.empty(T if reduction == "none" else 1, dtype=torch.float32, pin_memory=True)
        self.n_valid = int(np.sum(problem.labels != problem.ignore_index))
        # the forward call's kernels (forward_call_kernels) and the backward kernel
        self.launches_per_step = len(forward_call_kernels(V, T, self.es, reduction)) + 1

    def fwd(self, stream):
        if self.eps:
            self.vce.ce_forward_ls(self.logits, self.labels, self.eps, reduction=self.red, loss_rows=self.loss_rows,
                                   loss_out=self.loss_out, row_stats=self.stats, status=self.status, stream=stream)
        else:
            self.vce.ce_forward(self.logits, self.labels, reduction=self.red, loss_rows=self.loss_rows,
                                loss_out=self.loss_out, row_stats=self.stats, status=self.status, stream=stream)

    def bwd(self, stream):
        if self.eps:
            self.vce.ce_backward_ls(self.logits, self.labels, self.stats, self.go, self.eps, reduction=self.red,
                                    grad_logits=self.grad, stream=stream)
        else:
            self.vce.ce_backward(self.logits, self.labels, self.stats, self.go, reduction=self.red,
                                 grad_logits=self.grad, stream=stream)

    def step(self, stream):
        self.fwd(stream)
        self.bwd(stream)

    def one_pass_step(self, stream):
        """The same outputs through ce_forward_backward(_ls) (grad_output known before the forward)."""
        if self.eps:
            self.vce.ce_forward_backward_ls(self.logits, self.labels, self.eps, reduction=self.red,
                                            grad_output=self.go, grad_logits=self.grad, loss_rows=self.loss_rows,
                                            loss_out=self.loss_out, row_stats=self.stats, status=self.status,
                                            stream=stream)
        else:
            self.vce.ce_forward_backward(self.logits, self.labels, reduction=self.red, grad_output=self.go,
                                         grad_logits=self.grad, loss_rows=self.loss_rows, loss_out=self.loss_out,
                                         row_stats=self.stats, status=self.status, stream=stream)

    def e2e_step(self, stream):
        self.logits.copy_(self.host_bf16, non_blocking=True)
        self.labels.copy_(self.labels_host, non_blocking=True)
        self.step(stream)
        self.loss_host.copy_(self.loss_rows if self.red == "none" else self.loss_out, non_blocking=True)

    @property
    def h2d_bytes(self):
        return self.p.T * self.p.V * self.es + self.p.T * 8 + (self.p.T * 4 if self.red == "none" else 0)

    @property
    def d2h_bytes(self):
        return 4 * self.loss_host.numel()

    def tokens(self):
        return self.p.T

    def bytes_fwd(self):
        T, V = self.p.T, self.p.V
        return self.n_valid * V * self.es + T * (8 + 4 + 16)

    def bytes_bwd(self):
        T, V = self.p.T, self.p.V
        return self.n_valid * V * self.es + T * V * self.es + T * (8 + 16) + (T * 4 if self.red == "none" else 0)

    def describe(self):
        p = self.p
        red = {"mean": "mean over non-ignored rows", "sum": "sum over rows",
               "none": "per-row losses, per-row grad_output"}[self.red]
        return {"workload": f"{p.name}: CE fwd+bwd, T={p.T} rows x V={p.V} {p.dtype} logits, {red}, "
                            f"{len(p.margin_rows)} raised-target rows, {len(p.ignore_rows)} ignored",
                "T": p.T, "V": p.V, "logits": p.dtype, "grad": p.dtype, "math": "f32", "reduction": self.red,
                "label_smoothing": self.eps,
                "l2": "no flush: inputs (%.2f GB logits) larger than the 129 MB L2" % (p.T * p.V * self.es / 1e9)}


def backward_kernel(V):
    """The kernel ce_backward runs for contiguous, 16-byte aligned [T, V] logits and gradient."""
    return "k_ce_bwd_ring" if V % 8 == 0 else "k_ce_bwd"


BWD_RING_FILES = ["vocab_cross_entropy_gb300/csrc/ce_bwd_ring.cu", "vocab_cross_entropy_gb300/csrc/ce_stage.cuh",
                  "vocab_cross_entropy_gb300/csrc/ce_slots.cuh", "vocab_cross_entropy_gb300/csrc/vce_device.cuh",
                  "vocab_cross_entropy_gb300/csrc/vce_async.cuh"]


def forward_kernel(V, T=None, es=2):
    """The kernel ce_forward runs for contiguous, 16-byte aligned [T, V] logits: one warp per row
    for rows of at most 32 KB, the stage ring for longer rows (and one block per row for layouts
    neither takes)."""
    if V * es <= 32768:
        return "k_ce_fwd_warp"
    if V % 8:
        return "k_ce_fwd"
    return "k_ce_fwd_ring"


def forward_reduces_in_kernel(V, T, es, reduction):
    """Whether the ce_forward call's row kernel reduces the losses itself (the stage ring, SUM or
    MEAN, at most 65536 rows) instead of a k_ce_reduce launch after it."""
    return forward_kernel(V, T, es) == "k_ce_fwd_ring" and reduction != "none" and T <= 65536


def forward_call_kernels(V, T, es, reduction):
    """The ce_forward call's kernels in launch order: the row kernel, and k_ce_reduce unless the
    row kernel reduces the losses itself (or reduction is none).  The stage ring writes the status
    word itself; before the other row kernels a memset clears it (not a kernel of this library)."""
    k = forward_kernel(V, T, es)
    if reduction == "none":
        return [k]
    if forward_reduces_in_kernel(V, T, es, reduction):
        return [k + " (the loss reduction folded in)"]
    return [k, "k_ce_reduce"]


FWD_RING_FILES = ["vocab_cross_entropy_gb300/csrc/ce_fwd_ring.cu", "vocab_cross_entropy_gb300/csrc/ce_stage.cuh",
                  "vocab_cross_entropy_gb300/csrc/ce_fold.cuh", "vocab_cross_entropy_gb300/csrc/ce_slots.cuh",
                  "vocab_cross_entropy_gb300/csrc/vce_device.cuh", "vocab_cross_entropy_gb300/csrc/vce_async.cuh"]


CHUNK_FILES = ["vocab_cross_entropy_gb300/csrc/ce_fwd.cu", "vocab_cross_entropy_gb300/csrc/ce_rows.cuh",
               "vocab_cross_entropy_gb300/csrc/ce_bwd_ring.cu", "vocab_cross_entropy_gb300/csrc/ce_stage.cuh",
               "vocab_cross_entropy_gb300/csrc/ce_slots.cuh", "vocab_cross_entropy_gb300/csrc/ce_segments.h",
               "vocab_cross_entropy_gb300/csrc/vce_device.cuh", "vocab_cross_entropy_gb300/csrc/vce_async.cuh"]


def one_pass_kernel(V):
    """The kernel ce_forward_backward runs for contiguous, 16-byte aligned [T, V] buffers."""
    return "k_ce_fused_ring" if V % 8 == 0 else "k_ce_fused"


def one_pass_call_kernels(V, T, reduction):
    """The kernels of one ce_forward_backward call: the ring kernel counts N and reduces the losses
    itself for SUM / MEAN over at most 65536 rows; otherwise k_ce_count_valid (MEAN) comes first
    and k_ce_reduce (SUM / MEAN) last."""
    k = one_pass_kernel(V)
    if reduction == "none" or (k == "k_ce_fused_ring" and T <= 65536):
        return [k + (" (the loss reduction folded in)" if reduction != "none" else "")]
    return (["k_ce_count_valid"] if reduction == "mean" else []) + [k, "k_ce_reduce"]


class FusedWorkload(CEWorkload):
    """The pages' shape through ce_forward_backward: one pass over the logits per step."""

    def __init__(self, problem, device, reduction="mean"):
        super().__init__(problem, device, reduction)
        self.kernel = one_pass_kernel(problem.V)
        self.launches_per_step = len(one_pass_call_kernels(problem.V, problem.T, reduction))

    def step(self, stream):
        self.vce.ce_forward_backward(self.logits, self.labels, reduction=self.red, grad_output=self.go,
                                     grad_logits=self.grad, loss_rows=self.loss_rows, loss_out=self.loss_out,
                                     row_stats=self.stats, status=self.status, stream=stream)

    def bytes_fused(self):
        T, V = self.p.T, self.p.V
        return self.n_valid * V * self.es + T * V * self.es + T * (8 + 4 + 16 + 8)

    def describe(self):
        d = super().describe()
        d["workload"] = d["workload"].replace("CE fwd+bwd", "CE fwd+bwd in one pass (ce_forward_backward)")
        return d


class ChunkedWorkload(CEWorkload):
    """The pages' matrix as 8 column chunks in separate buffers: one ce_merge_chunks call per step."""

    def __init__(self, problem, device, reduction="mean"):
        super().__init__(problem, device, reduction)
        bounds = gen.chunk_bounds(problem.V, gen.CHUNKS)
        self.chunks = [self.logits[:, o:o + w].contiguous() for o, w in bounds]
        self.grads = [torch.empty_like(c) for c in self.chunks]
        del self.grad
        self.logits = None
        self.cstats = torch.empty(len(self.chunks), problem.T, 4, dtype=torch.float32, device=device)
        self.launches_per_step = 4            # k_ce_chunk_fwd, k_ce_merge, k_ce_reduce, k_ce_bwd

    def step(self, stream):
        self.vce.ce_merge_chunks(self.chunks, self.labels, reduction=self.red, grad_output=self.go,
                                 chunk_grads=self.grads,
                                 loss_rows=self.loss_rows, loss_out=self.loss_out, row_stats=self.stats,
                                 chunk_stats=self.cstats, status=self.status, stream=stream)

    def e2e_step(self, stream):
        for c, o_w in zip(self.chunks, gen.chunk_bounds(self.p.V, gen.CHUNKS)):
            o, w = o_w
            c.copy_(self.host_bf16[:, o:o + w], non_blocking=True)
        self.labels.copy_(self.labels_host, non_blocking=True)
        self.step(stream)
        self.loss_host.copy_(self.loss_out, non_blocking=True)

    def describe(self):
        d = super().describe()
        d["workload"] = d["workload"].replace("CE fwd+bwd", f"CE fwd+bwd over {gen.CHUNKS} column chunks of "
                                                            f"{gen.CHUNK_WIDTH} in separate buffers")
        return d


class LinearWorkload:
    """Fused linear-CE: E [8192, 4096], W [128256, 4096] bf16; one linear_ce_fwd_bwd call per step
    (linear_ce_fwd_bwd_filtered when filter_eps > 0)."""

    def __init__(self, problem, device, filter_eps=0.0):
        import vocab_cross_entropy_gb300 as vce
        self.vce = vce
        self.p = problem
        self.filter_eps = float(filter_eps)
        T, D, V = problem.T, problem.D, problem.V
        self.W_host = torch.empty((V, D), dtype=torch.int16, pin_memory=True)
        problem.W(out=self.W_host.numpy().view(np.uint16))
        self.E_host = torch.empty((T, D), dtype=torch.int16, pin_memory=True)
        problem.E(out=self.E_host.numpy().view(np.uint16), W=self.W_host.numpy().view(np.uint16))
        self.kept = torch.zeros(1, dtype=torch.int64, device=device)
        self.blocks = (-(-T // 128)) * (-(-V // 128))
        self.E = self.E_host.view(torch.bfloat16).to(device)
        self.W = self.W_host.view(torch.bfloat16).to(device)
        self.labels_host = torch.from_numpy(problem.labels).pin_memory()
        self.labels = self.labels_host.to(device)
        self.dE = torch.empty((T, D), dtype=torch.bfloat16, device=device)
        self.dW = torch.empty((V, D), dtype=torch.bfloat16, device=device)
        self.ws = torch.empty(vce.linear_ce_workspace_bytes(T, D, V), dtype=torch.uint8, device=device)
        self.loss_rows = torch.empty(T, dtype=torch.float32, device=device)
        self.loss_out = torch.empty(1, dtype=torch.float32, device=device)
        self.status = torch.empty(1, dtype=torch.int32, device=device)
        self.go = torch.ones(1, dtype=torch.float32, device=device)
        self.loss_host = torch.empty(1, dtype=torch.float32, pin_memory=True)
        nchunks = -(-V // 32768)
        # statistics GEMM + merge + reduce; per chunk the gradient-tile GEMM, dW (two launches over the
        # halves of T, or one over the kept blocks when filtering) and dE
        self.launches_per_step = 3 + (3 if filter_eps > 0 else 4) * nchunks

    def step(self, stream):
        if self.filter_eps > 0:
            self.vce.linear_ce_fwd_bwd_filtered(self.E, self.W, self.labels, self.filter_eps, grad_output=self.go,
                                                dE=self.dE, dW=self.dW, loss_rows=self.loss_rows,
                                                loss_out=self.loss_out, workspace=self.ws, kept_blocks=self.kept,
                                                status=self.status, stream=stream)
            return
        self.vce.linear_ce_fwd_bwd(self.E, self.W, self.labels, grad_output=self.go, dE=self.dE, dW=self.dW,
                                   loss_rows=self.loss_rows, loss_out=self.loss_out, workspace=self.ws,
                                   status=self.status, stream=stream)

    def timed_step(self, stream):
        """One call through linear_ce_fwd_bwd_timed: {GEMM kind: (milliseconds, launches)}."""
        _, split = self.vce.linear_ce_fwd_bwd_timed(self.E, self.W, self.labels, self.filter_eps,
                                                    grad_output=self.go, dE=self.dE, dW=self.dW,
                                                    loss_rows=self.loss_rows, loss_out=self.loss_out,
                                                    workspace=self.ws, kept_blocks=self.kept, status=self.status,
                                                    stream=stream)
        return split

    def full_size(self):
        """The shapes the committed GEMM captures were scaled to."""
        p = self.p
        return (p.T, p.D, p.V, self.filter_eps) == (8192, 4096, 128256, 0.0)

    def gemm_flops(self, kind):
        """(algorithmic, executed) flop of one call's GEMMs of a kind: z over all of [T, V] for
        the statistics and gradient-tile GEMMs; dW and dE over the kept 128 x 128 blocks of G
        (all of them without filtering), executed twice (G's hi and lo halves)."""
        p = self.p
        if kind in ("statistics", "gradient_tiles"):
            f = 2.0 * p.T * p.V * p.D
            return f, f
        f = 2.0 * p.T * p.V * p.D if self.filter_eps <= 0 else 2.0 * self.kept_blocks() * 128 * 128 * p.D
        return f, 2.0 * f

    def e2e_step(self, stream):
        self.E.copy_(self.E_host.view(torch.bfloat16), non_blocking=True)
        self.W.copy_(self.W_host.view(torch.bfloat16), non_blocking=True)
        self.labels.copy_(self.labels_host, non_blocking=True)
        self.step(stream)
        self.loss_host.copy_(self.loss_out, non_blocking=True)

    @property
    def h2d_bytes(self):
        p = self.p
        return (p.T + p.V) * p.D * 2 + p.T * 8

    d2h_bytes = 4

    def tokens(self):
        return self.p.T

    def kept_blocks(self):
        return int(self.kept.item()) if self.filter_eps > 0 else self.blocks

    def flops(self):
        """Algorithmic: z twice (statistics, then recomputed for G) over all of [T, V], and dE, dW
        over the kept 128 x 128 blocks of G (all of them without filtering)."""
        p = self.p
        if self.filter_eps <= 0:
            return 8.0 * p.T * p.V * p.D
        return 4.0 * p.T * p.V * p.D + 4.0 * self.kept_blocks() * 128 * 128 * p.D

    def executed_flops(self):
        """What the tensor cores run: G enters dE and dW as two bf16 halves (hi + lo)."""
        p = self.p
        if self.filter_eps <= 0:
            return 12.0 * p.T * p.V * p.D
        return 4.0 * p.T * p.V * p.D + 8.0 * self.kept_blocks() * 128 * 128 * p.D

    def describe(self):
        p = self.p
        d = {"workload": f"{p.name}: fused linear-CE fwd+bwd, E [{p.T}, {p.D}] x W [{p.V}, {p.D}] bf16, mean over "
                         f"non-ignored rows ({len(p.ignore_rows)} ignored), dE and dW bf16",
             "T": p.T, "D": p.D, "V": p.V, "operands": "bf16", "accumulate": "f32",
             "l2": "no flush: W (%.2f GB) larger than the 129 MB L2" % (p.V * p.D * 2 / 1e9)}
        if p.peak > 0:
            d["hidden_states"] = (f"aligned with their targets: E_i = {p.e_std} N(0,1) + a W_(t_i), target logit "
                                  f"~{p.peak} above the rest (a stand-in for a trained model's concentrated softmax)")
        if self.filter_eps > 0:
            k = self.kept_blocks()
            d.update(filter_eps=self.filter_eps, kept_blocks=k, blocks=self.blocks,
                     kept_fraction=round(k / self.blocks, 5))
        return d


# ------------------------------------------------------------------------------- timing

def time_steps(fn, steps, stream, world, device, per_launch=None):
    """Time `steps` calls of fn(stream) with CUDA events on `stream`; max over ranks."""
    barrier(world)
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn(stream)
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize(device)
    barrier(world)
    ms = start.elapsed_time(end)
    return max_over_ranks(ms, world, device)


def time_kernel(workload, steps, stream):
    """Average duration of the forward and backward launches, events on the launching stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b, c in evs:
        a.record(stream)
        workload.fwd(stream)
        b.record(stream)
        workload.bwd(stream)
        c.record(stream)
    torch.cuda.synchronize()
    f = [a.elapsed_time(b) for a, b, _ in evs]
    g = [b.elapsed_time(c) for _, b, c in evs]
    return statistics.mean(f), statistics.mean(g)


def cpu_oracle_baseline(problem, budget_s=8.0):
    """The fp64 oracle as it stands, on a row sample of the same workload (host cores): once on
    one core, then on every core at once (one fresh worker process per core, each on its own
    share of the sample; started with subprocess, never forked from this CUDA process)."""
    from oracle import cpu_timing
    one = cpu_timing.time_rows(problem, 0, 1, budget_s)
    single = one["rows"] / (one["stop"] - one["start"])
    cores = os.cpu_count() or 1
    spec = json.dumps({k: getattr(problem, k) for k in ("name", "T", "V", "dtype", "seed", "std", "n_margin",
                                                       "margin_lo", "margin_hi", "n_ignore")})
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    procs = [subprocess.Popen([sys.executable, "-m", "oracle.cpu_timing", spec, str(i), str(cores), str(budget_s)],
                              cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
             for i in range(cores)]
    parts = []
    for pr in procs:
        out, _ = pr.communicate(timeout=budget_s + 120)
        if pr.returncode == 0 and out.strip():
            parts.append(json.loads(out.strip().splitlines()[-1]))
    rec = {"value": single, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{one['rows']} random rows of the same T={problem.T}, V={problem.V} matrix (input generation "
                     f"included), fp64 numpy forward+backward on one core, {one['stop'] - one['start']:.1f} s",
           "host_cores": cores}
    if len(parts) == cores:
        rows = sum(p_["rows"] for p_ in parts)
        wall = max(p_["stop"] for p_ in parts) - min(p_["start"] for p_ in parts)
        rec.update(value=rows / wall, cores=cores,
                   sample=f"{rows} random rows of the same T={problem.T}, V={problem.V} matrix (input generation "
                          f"included), fp64 numpy forward+backward, {cores} worker processes (one per host core, "
                          f"one thread each) for {wall:.1f} s",
                   single_core={"value": single, "cores": 1, "rows": one["rows"],
                                "seconds": round(one["stop"] - one["start"], 2)})
    else:
        rec["all_cores"] = f"unavailable: {len(parts)} of {cores} worker processes reported"
    return rec


def cpu_oracle_baseline_linear(problem, budget_s=12.0, max_rows=256):
    """The fp64 linear-CE oracle as it stands on a row sample (host cores): z over the whole
    vocabulary, the loss, G and the dE row of each sampled row; W widened once, untimed."""
    from oracle import ce_oracle as O
    W = O.widen(problem.W(), "bf16")
    N = int(np.sum(problem.labels != problem.ignore_index))
    order = np.random.default_rng(123).permutation(problem.T)
    done, block = 0, 2
    t0 = time.perf_counter()
    while done < max_rows and time.perf_counter() - t0 < budget_s:
        rows = np.sort(order[done: done + block])
        E = O.widen(problem.E_rows(rows), "bf16")
        z = E @ W.T
        fwd = O.ce_rows(z, problem.labels[rows])
        G = O.ce_grad_rows(z, problem.labels[rows], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
        G @ W
        done += len(rows)
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or os.cpu_count() or 1)
    return {"value": done / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} random rows of the same T={problem.T}, D={problem.D}, V={problem.V} problem: z over "
                      f"all columns, loss, G and the dE row, fp64 numpy (matrix products on up to {cores} BLAS "
                      f"threads), {dt:.1f} s; W widened once, untimed"}


# ------------------------------------------------------------------------------- main

def linear_problem(args, rank, peaked):
    problem = gen.linear_peaked(seed=1006 + rank) if peaked else gen.linear(seed=1005 + rank)
    if args.vocab:
        problem = gen.LinearProblem(f"{problem.name}[V={args.vocab}]", problem.T, problem.D, args.vocab,
                                    problem.seed, problem.n_ignore, problem.e_std, problem.w_std, problem.peak)
    return problem


LINEAR_GEMMS = {
    "statistics": "k_tc_gemm<EpiStats> (z = E W^T, per-tile row statistics)",
    "gradient_tiles": "k_tc_gemm<EpiGrad> (z recomputed, G = c (p - onehot) as bf16 hi + lo)",
    "dW": "k_tc_gemm<EpiKahan> (dW = G^T E over the halves of T, two-sum merge; G_hi and G_lo tiles beside one E tile)",
    "dE": "k_tc_gemm<EpiKahan> (dE += G W, two-sum across chunks; G_hi and G_lo tiles beside one W tile)",
}


def measure_linear(w, steps, warmup, e2e_steps, world, device, local_rank):
    """Times linear-CE calls (CUDA events on the launching stream), the per-GEMM split of one
    call (events around each GEMM launch), and the end-to-end call with host copies."""
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        w.step(stream)
    torch.cuda.synchronize(device)
    with ClockSampler(local_rank) as clk:
        ms = time_steps(w.step, steps, stream, world, device)
    clocks = clk.summary()
    # per-GEMM split: a few timed calls (blocking), averaged
    reps = max(3, min(steps, 10))
    tot = {k: [0.0, 0] for k in LINEAR_GEMMS}
    for _ in range(reps):
        split = w.timed_step(stream)
        for k, (m, n) in split.items():
            tot[k][0] += m / reps
            tot[k][1] = n
    e2e_steps = max(3, min(e2e_steps, steps))
    w.e2e_step(stream)
    e2e_ms = time_steps(w.e2e_step, e2e_steps, stream, world, device)
    status = w.vce.vce_get_status(w.status)
    if status != 0:
        raise RuntimeError(f"device status {status}")
    return {"ms_step": ms / steps, "e2e_ms": e2e_ms / e2e_steps, "e2e_steps": e2e_steps, "clocks": clocks,
            "gemms": tot, "tokens_all": sum_over_ranks(w.tokens(), world, device)}


def linear_record(w, m, peaks, world):
    """The linear-CE measurement as a JSON object: throughput, tensor-core rate against the
    measured bf16 peaks (burst as `frac`, sustained beside it), the per-GEMM split with the
    dominant GEMM's roofline, clocks and the end-to-end figure."""
    ms = m["ms_step"]
    alg = w.flops() / (ms / 1e3) / 1e12
    exe = w.executed_flops() / (ms / 1e3) / 1e12
    gemms = {}
    for k, (gms, n) in m["gemms"].items():
        fa, fe = w.gemm_flops(k)
        gemms[k] = {"kernel": LINEAR_GEMMS[k], "launches": n, "ms_per_call": round(gms, 4),
                    "ms_per_launch": round(gms / max(n, 1), 4),
                    "algorithmic_tflops": round(fa / (gms / 1e3) / 1e12, 1) if gms > 0 else None,
                    "executed_tflops": round(fe / (gms / 1e3) / 1e12, 1) if gms > 0 else None}
    dom = max(gemms, key=lambda k: gemms[k]["ms_per_call"])
    d = gemms[dom]
    return {
        "value": round(m["tokens_all"] / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_call": round(ms, 4),
        "algorithmic_tflops": round(alg, 1), "executed_tflops": round(exe, 1),
        "frac": round(alg / peaks["bf16_tflops"], 4), "peak": peaks["bf16_tflops"],
        "frac_of_sustained": round(alg / peaks["bf16_tflops_sustained"], 4),
        "peak_sustained": peaks["bf16_tflops_sustained"], "peak_source": peaks["source"],
        "algorithmic_flop_per_call": w.flops(), "executed_flop_per_call": w.executed_flops(),
        "gemms": gemms,
        "roofline": {"bound": "tensor", "kernel": d["kernel"], "achieved": d["algorithmic_tflops"],
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(d["algorithmic_tflops"] / peaks["bf16_tflops"], 4),
                     "executed": d["executed_tflops"], "ms_per_launch": d["ms_per_launch"],
                     "traffic": profiled_traffic(f"linear_{dom}_gemm", LINEAR_FILES) if w.full_size() else None},
        "e2e": {"value": round(m["tokens_all"] / (m["e2e_ms"] / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": w.h2d_bytes, "d2h_bytes_per_step": w.d2h_bytes, "steps": m["e2e_steps"]},
        "gpu_launches_per_call": w.launches_per_step,
        "clocks": m["clocks"],
    }


LINEAR_FILES = ["vocab_cross_entropy_gb300/csrc/lce.cu", "vocab_cross_entropy_gb300/csrc/tc_gemm.cuh",
                "vocab_cross_entropy_gb300/csrc/tc_launch.cuh", "vocab_cross_entropy_gb300/csrc/vce_async.cuh",
                "vocab_cross_entropy_gb300/csrc/vce_device.cuh", "vocab_cross_entropy_gb300/csrc/vce_check.cuh"]


def run_linear(args, rank, local_rank, world, device):
    peaked = args.workload == "linear_peaked"
    problem = linear_problem(args, rank, peaked)
    eps = args.filter_eps if args.filter_eps is not None else (2.0 ** -12 if peaked else 0.0)
    w = LinearWorkload(problem, device, eps)
    m = measure_linear(w, args.steps, args.warmup, args.e2e_steps, world, device, local_rank)
    peaks = measured_peaks()
    rec = linear_record(w, m, peaks, world)
    call = "linear_ce_fwd_bwd_filtered" if eps > 0 else "linear_ce_fwd_bwd"
    out = {
        "metric": ("fused linear-CE fwd+bwd tokens/s at T=8192, D=4096, V=128256 bf16"
                   + (f", gradient filtering at eps={eps:.3g}" if eps > 0 else "") + "; TFLOP/s vs bf16 peak"),
        "value": rec["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_call"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(w.describe(), parallelism=f"replicas{world}", call=call),
        "roofline": rec["roofline"],
        "call_tflops": {k: rec[k] for k in ("algorithmic_tflops", "executed_tflops", "frac", "peak",
                                            "frac_of_sustained", "peak_sustained", "peak_source")},
        "gemms": rec["gemms"],
        "e2e": rec["e2e"],
        "gpu_launches": w.launches_per_step * args.steps,
        "clocks": rec["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_oracle_baseline_linear(problem)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_ours(args, rank, local_rank, world):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    if args.workload in ("linear", "linear_peaked"):
        return run_linear(args, rank, local_rank, world, device)
    problem = {"pages": gen.pages, "chunked": gen.pages, "fused": gen.pages, "mid": gen.mid}[args.workload](
        seed=(1002 if args.workload == "mid" else 1003) + rank)
    if args.logits_dtype != problem.dtype:
        problem = gen.CEProblem(problem.name, problem.T, problem.V, args.logits_dtype, problem.seed, problem.std,
                                problem.n_margin, problem.margin_lo, problem.margin_hi, problem.n_ignore)
    if args.rows:
        problem = gen.CEProblem(problem.name + f"[{args.rows} rows]", args.rows, problem.V, problem.dtype,
                                problem.seed, problem.std, round(0.10 * args.rows) if problem.n_margin else 0,
                                problem.margin_lo, problem.margin_hi, round(problem.n_ignore * args.rows / problem.T))
    if args.label_smoothing and args.workload != "pages":
        raise SystemExit("--label-smoothing applies to the pages workload (ce_forward_ls / ce_backward_ls)")
    if args.label_smoothing:
        w = CEWorkload(problem, device, args.reduction, args.label_smoothing)
    else:
        w = {"chunked": ChunkedWorkload, "fused": FusedWorkload}.get(args.workload, CEWorkload)(problem, device,
                                                                                            args.reduction)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        w.step(stream)
    torch.cuda.synchronize(device)
    with ClockSampler(local_rank) as clk:
        ms = time_steps(w.step, args.steps, stream, world, device)
    clocks = clk.summary()
    chunked = args.workload in ("chunked", "fused")
    if not chunked:
        fwd_ms, bwd_ms = time_kernel(w, max(10, min(args.steps, 50)), stream)
        # the forward call alone, back to back (no backward's dirty L2 written back under it)
        for _ in range(3):
            w.fwd(stream)
        fwd_alone_ms = time_steps(w.fwd, args.steps, stream, world, device) / args.steps
        for _ in range(3):
            w.one_pass_step(stream)
        one_pass_ms = time_steps(w.one_pass_step, args.steps, stream, world, device) / args.steps
    e2e_steps = max(3, min(args.e2e_steps, args.steps))
    for _ in range(2):
        w.e2e_step(stream)
    e2e_ms = time_steps(w.e2e_step, e2e_steps, stream, world, device)
    status = w.vce.vce_get_status(w.status)
    if status != 0:
        raise RuntimeError(f"device status {status}")

    tokens_all = sum_over_ranks(w.tokens(), world, device)
    ms_step = ms / args.steps
    value = tokens_all / (ms_step / 1e3)
    e2e_value = tokens_all / (e2e_ms / e2e_steps / 1e3)
    peaks = measured_peaks()
    bwd_bytes = w.bytes_bwd()
    if args.workload == "fused":   # one call: the fused kernel plus two one-block kernels
        call_bytes = w.bytes_fused()
        achieved = call_bytes / (ms_step / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "ce_forward_backward (" + " + ".join(one_pass_call_kernels(w.p.V, w.p.T, w.red)) + ")",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": call_bytes,
                "traffic": profiled_traffic("k_ce_fused_ring_pages", RING_FILES) if captured_shape(w) else None}
    elif chunked:   # one call launches all four kernels: roofline over the whole call
        call_bytes = w.bytes_fwd() + bwd_bytes + 2 * w.p.T * gen.CHUNKS * 16
        achieved = call_bytes / (ms_step / 1e3) / 1e9
        ring = all(wd % 8 == 0 for _, wd in gen.chunk_bounds(w.p.V, gen.CHUNKS))
        roof = {"bound": "hbm", "kernel": "ce_merge_chunks (k_ce_chunk_fwd + k_ce_merge + k_ce_reduce + "
                                          + ("k_ce_bwd_ring" if ring else "k_ce_bwd") + ")",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                "algorithmic_bytes_per_launch": call_bytes,
                "traffic": (profiled_traffic("ce_merge_chunks_pages", CHUNK_FILES)
                            if args.workload == "chunked" and ring and captured_shape(w) else None)}
    else:
        achieved = bwd_bytes / (bwd_ms / 1e3) / 1e9
        bkern = backward_kernel(w.p.V)
        traffic = None
        if captured_shape(w):
            traffic = (profiled_traffic("k_ce_bwd_ring_pages", BWD_RING_FILES) if bkern == "k_ce_bwd_ring"
                       else profiled_traffic("k_ce_bwd_pages", CEWorkload.KERNEL_FILES))
        roof = {"bound": "hbm", "kernel": bkern, "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"], "algorithmic_bytes_per_launch": bwd_bytes, "traffic": traffic}
    out = {
        "metric": "CE fwd+bwd tokens/s at T=16384,V=128256 bf16; HBM GB/s vs ~8 TB/s",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(w.describe(), parallelism=f"replicas{world}"),
        "hbm_gbs_step": round((w.bytes_fused() if args.workload == "fused" else w.bytes_fwd() + bwd_bytes) * world
                              / (ms_step / 1e3) / 1e9, 1),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": w.h2d_bytes,
                "d2h_bytes_per_step": w.d2h_bytes, "steps": e2e_steps},
        "gpu_launches": w.launches_per_step * args.steps,
        "clocks": clocks,
    }
    if not chunked:
        out["kernels_ms"] = {"ce_forward": round(fwd_ms, 5), "ce_backward": round(bwd_ms, 5)}
        if one_pass_ms:
            one_bytes = (w.n_valid + w.p.T) * w.p.V * w.es
            one_gbs = one_bytes / (one_pass_ms / 1e3) / 1e9
            out["one_pass"] = {"call": "ce_forward_backward_ls" if w.eps else "ce_forward_backward",
                               "kernel": one_pass_kernel(w.p.V),
                               "value": round(tokens_all / (one_pass_ms / 1e3), 1), "unit": "tokens/s",
                               "ms_per_step": round(one_pass_ms, 5), "algorithmic_bytes_per_step": one_bytes,
                               "hbm_gbs": round(one_gbs, 1), "frac": round(one_gbs / peaks["hbm_gbs"], 4),
                               "traffic": (profiled_traffic("k_ce_fused_ring_pages", RING_FILES)
                                           if captured_shape(w) and one_pass_kernel(w.p.V) == "k_ce_fused_ring"
                                           else None)}
        fkern = forward_kernel(w.p.V, w.p.T, w.es)
        out["roofline_fwd"] = {"bound": "hbm", "kernel": " + ".join(forward_call_kernels(w.p.V, w.p.T, w.es, w.red)) + " (the ce_forward call)",
                               "achieved": round(w.bytes_fwd() / (fwd_ms / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                               "unit": "GB/s",
                               "frac": round(w.bytes_fwd() / (fwd_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                               "back_to_back": {"ms": round(fwd_alone_ms, 5),
                                                "frac": round(w.bytes_fwd() / (fwd_alone_ms / 1e3) / 1e9
                                                              / peaks["hbm_gbs"], 4)},
                               "traffic": (profiled_traffic("k_ce_fwd_ring_pages", FWD_RING_FILES)
                                           if captured_shape(w) and fkern == "k_ce_fwd_ring" else None)}
    if args.workload == "pages" and not args.no_linear and not args.rows and args.logits_dtype == "bf16" \
            and args.reduction == "mean" and not args.label_smoothing:
        # the fused linear-CE of the same run (E [8192, 4096], W [128256, 4096] bf16) beside the CE line
        del w
        torch.cuda.empty_cache()
        lw = LinearWorkload(linear_problem(args, rank, False), device, 0.0)
        lm = measure_linear(lw, min(args.steps, 30), args.warmup, args.e2e_steps, world, device, local_rank)
        lsteps = min(args.steps, 30)
        out["linear"] = dict(linear_record(lw, lm, peaks, world), call="linear_ce_fwd_bwd",
                             workload=lw.describe()["workload"], steps=lsteps,
                             gpu_launches=lw.launches_per_step * lsteps)
        del lw
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_oracle_baseline(problem)
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference_linear(args, world):
    """The linear-CE oracle (fp64, CPU) on sampled rows: z, loss and G for each row over the whole
    vocabulary, and its dE row.  W is widened once, outside the timed steps; dW needs every
    row and is not sampled.  The filtered workload's rows are timed unfiltered (the filter's
    block decisions need 128 rows of z per sampled row)."""
    from oracle import ce_oracle as O
    peaked = args.workload == "linear_peaked"
    p = gen.linear_peaked() if peaked else gen.linear()
    if args.vocab:
        p = gen.LinearProblem(f"{p.name}[V={args.vocab}]", p.T, p.D, args.vocab, p.seed, p.n_ignore, p.e_std,
                              p.w_std, p.peak)
    W = O.widen(p.W(), "bf16")
    N = int(np.sum(p.labels != p.ignore_index))
    rows_per_step = 2
    rng = np.random.default_rng(7)

    def one_step():
        rows = np.sort(rng.choice(p.T, rows_per_step, replace=False))
        E = O.widen(p.E_rows(rows), "bf16")
        z = E @ W.T
        fwd = O.ce_rows(z, p.labels[rows])
        G = O.ce_grad_rows(z, p.labels[rows], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
        return G @ W

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    eps = args.filter_eps if args.filter_eps is not None else (2.0 ** -12 if peaked else 0.0)
    metric = ("fused linear-CE fwd+bwd tokens/s at T=8192, D=4096, V=128256 bf16"
              + (f", gradient filtering at eps={eps:.3g}" if eps > 0 else "") + "; TFLOP/s vs bf16 peak")
    # the row products go through numpy's BLAS, which runs on every host core unless told otherwise
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or os.cpu_count() or 1)
    sample = (f"{rows_per_step} random rows per step: z over all {p.V} columns, loss, G and the dE row, "
              f"fp64 numpy, matrix products on up to {cores} BLAS threads" + (", unfiltered" if eps > 0 else ""))
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{p.name}: fused linear-CE T={p.T} D={p.D} V={p.V}, {rows_per_step} sampled rows "
                               "per step", "T": p.T, "D": p.D, "V": p.V},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args, rank, world):
    """The oracle (fp64, CPU) as the reference arm: rank 0 alone, bounded samples per step."""
    if rank != 0:
        return
    if args.workload in ("linear", "linear_peaked"):
        return run_reference_linear(args, world)
    # the one-pass and chunked workloads hold the pages' matrix
    problem = {"pages": gen.pages, "fused": gen.pages, "chunked": gen.pages, "mid": gen.mid}[args.workload]()
    from oracle import ce_oracle as O
    N = int(np.sum(problem.labels != problem.ignore_index))
    rows_per_step = 64
    rng = np.random.default_rng(7)

    def one_step():
        rows = np.sort(rng.choice(problem.T, rows_per_step, replace=False))
        z = O.widen(problem.rows(rows), problem.dtype)
        fwd = O.ce_rows(z, problem.labels[rows])
        O.ce_grad_rows(z, problem.labels[rows], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    out = {
        "impl": "reference", "metric": "CE fwd+bwd tokens/s at T=16384,V=128256 bf16; HBM GB/s vs ~8 TB/s",
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{problem.name}: CE fwd+bwd T={problem.T} V={problem.V} bf16 logits, "
                               f"{rows_per_step} sampled rows per step", "T": problem.T, "V": problem.V},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} random rows per step of the same matrix, fp64 numpy"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["pages", "fused", "chunked", "mid", "linear", "linear_peaked"],
                    default="pages")
    ap.add_argument("--filter-eps", type=float, default=None,
                    help="linear workloads: gradient-filter threshold (default 2^-12 for linear_peaked, 0 for linear)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--logits-dtype", choices=["bf16", "f32"], default="bf16",
                    help="storage type of the logits (and gradient) for the CE workloads")
    ap.add_argument("--reduction", choices=["mean", "sum", "none"], default="mean")
    ap.add_argument("--label-smoothing", type=float, default=0.0,
                    help="pages workload through ce_forward_ls / ce_backward_ls with this eps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-linear", action="store_true",
                    help="pages workload: leave out the fused linear-CE record of the default line")
    ap.add_argument("--rows", type=int, default=None,
                    help="profiling only: draw the first ROWS rows of the workload instead of all T")
    ap.add_argument("--vocab", type=int, default=None,
                    help="profiling only: a smaller vocabulary for the linear workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local_rank, world = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
