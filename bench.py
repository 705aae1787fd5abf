"""Benchmark of the fused CE + TVD loss, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--rows BT]

One step = the whole hot path over one batch: the fused forward (two-pass
log-sum-exp, TVD and sigma) and the fused backward (gradient w.r.t. the
student logits), through the C ABI, on inputs already resident in HBM.
The workload's upstream gradients are per-row constants known before the
forward, so the headline step (``--path single``) is the single-launch
forward + backward; ``--path two`` times the separate forward and backward
launches, and each run also times the other path for comparison.  Both
write bit-identical outputs.  The default workload is BT = 8192 rows of
V = 151936 bf16 logits; a step streams at least 7.4 GB, far more than L2, so
L2 needs no flush between steps.

Under torchrun every rank runs the full per-rank workload on its own GPU
(rows are independent, so there is no collective on the data path) and
rank 0 prints one JSON line with the max-over-ranks time.

``--impl reference`` times the CPU fp64 oracle instead, on the host cores,
over a bounded sample of rows of the same workload each step.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from distillation_ce_tvd_gb300 import binding, sharding, vocab_parallel, workloads  # noqa: E402

METRIC = "fused CE+TVD fwd+bwd tokens/s and HBM GB/s (% of peak), V=151936 bf16, 1 GB300"
DEFAULT_WORKLOAD = "bt8192_v151936_bf16"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ["fct_common.cuh", "fct_forward.cu", "fct_backward.cu"]
# Algorithmic bytes per launch (per-row scalars ignored): the forward reads
# student + teacher once (2 V e per row); the backward and the single-launch
# forward + backward read both and write the gradient (3 V e per row).


# ---------------------------------------------------------------- helpers

def kernel_source_hash() -> str:
    """Hash of the kernels' code: comments and blank lines are left out, so a
    measured traffic figure stays attached to the code it was measured on."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "distillation_ce_tvd_gb300", "csrc", f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*$", "", line).strip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.cmd = ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                        "--format=csv,noheader,nounits", "-lms", "100"]
        except Exception:
            self.cmd = None

    def __enter__(self):
        if self.cmd:
            try:
                self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.3)
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle

def cpu_oracle_rate(w_rows, threads=None) -> tuple[float, float, int]:
    """(rows/s, seconds, threads) of the oracle's forward + backward on host rows."""
    import oracle
    oracle.build()
    n = threads or os.cpu_count() or 1
    s, t, tg = w_rows.student, w_rows.teacher, w_rows.target.numpy()
    t0 = time.perf_counter()
    oracle.fused_ce_tvd_forward(s, t, tg, w_rows.ignore_index, threads=n)
    oracle.fused_ce_tvd_backward(s, t, tg, w_rows.grad_ce.numpy(), w_rows.grad_tvd.numpy(),
                                 w_rows.ignore_index, threads=n)
    dt = time.perf_counter() - t0
    return w_rows.BT / dt, dt, n


def host_rows(name: str, rows: int, BT: int | None = None):
    """A bounded sample of the workload's rows, generated on the host."""
    return workloads.make(name, "cpu", rows=rows)


def cpu_model() -> str:
    """The host CPU's model name as the OS reports it."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def single_core_rate(name: str = "bt1024_v32000_bf16", seconds: float = 2.0) -> dict:
    """The oracle on one thread, on rows of a small workload, for scale."""
    probe = host_rows(name, 2)
    rate, _, _ = cpu_oracle_rate(probe, threads=1)
    rows = int(max(2, min(workloads.WORKLOADS[name]["BT"], rate * seconds)))
    rate, dt, _ = cpu_oracle_rate(host_rows(name, rows), threads=1)
    return {"workload": name, "rows": rows, "value": rate, "unit": "tokens/s", "seconds": dt}


def cpu_baseline(name: str, target_seconds: float = 12.0) -> dict:
    probe = host_rows(name, 8)
    rate, dt, n = cpu_oracle_rate(probe)
    rows = int(max(8, min(workloads.WORKLOADS[name]["BT"], rate * target_seconds)))
    sample = host_rows(name, rows)
    rate, dt, n = cpu_oracle_rate(sample)
    return {"value": rate, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{rows} rows of {name} (fwd+bwd, fp64, OpenMP over rows), {dt:.1f} s",
            "cpu_model": cpu_model(), "single_core": single_core_rate()}


# ---------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    name = args.workload
    cfg = workloads.WORKLOADS[name]
    probe = host_rows(name, 4)
    rate, _, n = cpu_oracle_rate(probe)
    total = max(1, args.steps + args.warmup)
    rows = int(max(1, min(cfg["BT"], rate * 150.0 / total)))
    sample = host_rows(name, rows)
    for _ in range(args.warmup):
        cpu_oracle_rate(sample, n)
    times = []
    for _ in range(args.steps):
        _, dt, _ = cpu_oracle_rate(sample, n)
        times.append(dt)
    sec = sum(times) / len(times)
    value = rows / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "BT": cfg["BT"], "V": cfg["V"],
                   "logit_dtype": "bf16" if cfg["dtype"] == torch.bfloat16 else "f32",
                   "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
                         "sample": f"{rows} rows of {name} per step (fwd+bwd, fp64)",
                         "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------- fused linear

def run_linear(args, world, rank, local):
    """Fused-linear CE + TVD: hidden states and lm_head weights in, the loss and
    the student's hidden and weight gradients out, logits only in row blocks.
    Dominated by four GEMMs per block (the library's tcgen05 GEMM)."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()
    w = workloads.make_linear(args.workload, dev, rows=args.rows)
    BT, ds = w.h_student.shape
    V, dt = w.w_teacher.shape
    rows = min(args.chunk_rows, BT)
    ldt = torch.bfloat16 if args.logits_dtype == "bf16" else torch.float32
    ws_bytes = binding.fused_linear_ce_tvd_workspace_size(V, rows, ldt)
    workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    grad_h = torch.empty_like(w.h_student)
    grad_w = torch.zeros(V, ds, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.fused_linear_ce_tvd_forward_backward(
            w.h_student, w.w_student, w.h_teacher, w.w_teacher, w.target, w.grad_ce, w.grad_tvd,
            w.ignore_index, chunk_rows=rows, logits_dtype=ldt, workspace=workspace,
            grad_h=grad_h, grad_w=grad_w,
            stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.__enter__()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        step()
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    if clocks:
        clocks.__exit__(None, None, None)
    ms = sharding.max_over_ranks(a.elapsed_time(b) / K, world, dev)
    flops = 2.0 * BT * V * (ds + dt) + 2.0 * 2.0 * BT * V * ds  # logits of both; d hidden, d weight
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(peaks_path))["bf16_tflops_sustained"] if os.path.exists(peaks_path) else 1700.0
    tflops = flops / (ms * 1e-3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": "fused-linear CE+TVD fwd+bwd tokens/s (GEMM-bound), 1 GB300",
            "value": world * BT / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "BT": BT, "V": V, "d_student": ds,
                       "d_teacher": dt, "chunk_rows": rows, "logits_dtype": args.logits_dtype,
                       "workspace_bytes": ws_bytes},
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak,
                         "unit": "TFLOP/s", "frac": tflops / peak, "traffic": None,
                         "peak_source": "measured cuBLAS bf16, sustained"},
            # per row block: two logit GEMMs, the loss kernel, d hidden, d weight
            "gpu_launches": K * ((BT + rows - 1) // rows) * 5,
            "clocks": clocks.summary() if clocks else None,
        }))


# ---------------------------------------------------------------- GEMM alone

GEMM_PRODUCTS = {
    # the fused-linear path's products for one row block of R rows
    "logits": "C (R x V, bf16) = H (R x D) W^T",
    "d_hidden": "C (R x D, bf16) = G (R x V) W (V x D), W read MN-major, split K",
    "d_weight": "C (V x D, fp32) += G^T (V x R) H (R x D), both MN-major",
}


def run_gemm(args):
    """Times one of the fused-linear path's GEMMs on the library's tcgen05
    kernel (profiling and tuning; not the headline)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load()
    R, D, V = (int(x) for x in args.gemm_shape.split(","))
    g = torch.Generator(device=dev).manual_seed(3)
    h = torch.randn(R, D, generator=g, device=dev).bfloat16()
    w = (torch.randn(V, D, generator=g, device=dev) * 0.03).bfloat16()
    G = (torch.randn(R, V, generator=g, device=dev) * 1e-4).bfloat16()
    if args.gemm == "logits":
        c = torch.empty(R, V, device=dev, dtype=torch.bfloat16)
        ws = None
        fn = lambda: binding.fct_gemm_bf16(h, w, c)  # noqa: E731
    elif args.gemm == "d_hidden":
        c = torch.empty(R, D, device=dev, dtype=torch.bfloat16)
        ws = torch.empty(binding.fct_gemm_bf16_workspace_size(R, D), device=dev,
                         dtype=torch.uint8)
        fn = lambda: binding.fct_gemm_bf16(G, w.t(), c, workspace=ws)  # noqa: E731
    else:
        c = torch.zeros(V, D, device=dev)
        fn = lambda: binding.fct_gemm_bf16(G.t(), h.t(), c, accumulate=True)  # noqa: E731
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / args.steps
    tflops = 2.0 * R * D * V / (ms * 1e-3) / 1e12
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(peaks_path))["bf16_tflops"] if os.path.exists(peaks_path) else 1900.0
    print(json.dumps({"gemm": args.gemm, "product": GEMM_PRODUCTS[args.gemm], "R": R, "D": D,
                      "V": V, "ms": ms, "tflops": tflops, "peak_burst": peak,
                      "frac": tflops / peak}))


# ---------------------------------------------------------------- our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.LINEAR_WORKLOADS))
    ap.add_argument("--chunk-rows", type=int, default=2048, help="row block of the fused-linear path")
    ap.add_argument("--logits-dtype", default="f32", choices=["f32", "bf16"],
                    help="element type of the fused-linear path's logit blocks")
    ap.add_argument("--rows", type=int, default=None, help="override BT (profiling)")
    ap.add_argument("--path", default="single", choices=["single", "two", "two_signs"],
                    help="headline step: one fused forward+backward launch, or the forward "
                         "and backward launches")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-block-rows", type=int, default=256,
                    help="row block of the host-buffer entry point")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-other", action="store_true", help="skip timing the other path")
    ap.add_argument("--cluster", type=int, default=0,
                    help="CTAs per row in the fused forward (0 = automatic)")
    ap.add_argument("--ring", type=int, default=0, choices=[0, 1, 2],
                    help="shared-memory staging of the multi-pass kernels: 0 automatic, "
                         "1 per-thread cp.async ring, 2 producer-warp TMA bulk-copy ring")
    ap.add_argument("--gemm", default=None, choices=sorted(GEMM_PRODUCTS),
                    help="time one fused-linear GEMM alone (R,D,V from --gemm-shape)")
    ap.add_argument("--gemm-shape", default="2048,4096,151936")
    args = ap.parse_args()

    if args.gemm:
        run_gemm(args)
        return
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit at once
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.workload in workloads.LINEAR_WORKLOADS:
        run_linear(args, world, rank, local)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()
    opts = binding.options(ctas_per_row=args.cluster, ring=args.ring)
    # the other staging of the single launch, timed beside the headline (the
    # automatic choice is the bulk-copy ring where a row belongs to one CTA)
    alt_ring = binding.RING_TMA if args.ring == binding.RING_CP_ASYNC else binding.RING_CP_ASYNC
    opts_alt = binding.options(ctas_per_row=args.cluster, ring=alt_ring)
    # each rank holds its own batch of the workload (weak scaling, no exchange)
    seed = workloads.WORKLOADS[args.workload]["seed"] + 1000 * rank
    w = workloads.make(args.workload, dev, rows=args.rows, seed=seed)
    BT, V = w.BT, w.V
    elem = w.student.element_size()
    ce = torch.empty(BT, device=dev)
    tvd = torch.empty_like(ce)
    ls = torch.empty_like(ce)
    lt = torch.empty_like(ce)
    sg = torch.empty_like(ce)
    grad = torch.empty_like(w.student)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        binding.fused_ce_tvd_forward(w.student, w.teacher, w.target, w.ignore_index, ce=ce, tvd=tvd,
                                     student_lse=ls, teacher_lse=lt, sigma=sg, stream=stream,
                                     options=opts)

    def bwd():
        binding.fused_ce_tvd_backward(w.student, w.teacher, w.target, ls, lt, sg, w.grad_ce,
                                      w.grad_tvd, w.ignore_index, grad_student=grad, stream=stream)

    def single():
        binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                              w.grad_tvd, w.ignore_index, ce=ce, tvd=tvd,
                                              student_lse=ls, teacher_lse=lt, sigma=sg,
                                              grad_student=grad, stream=stream, options=opts)

    def single_alt():
        binding.fused_ce_tvd_forward_backward(w.student, w.teacher, w.target, w.grad_ce,
                                              w.grad_tvd, w.ignore_index, ce=ce, tvd=tvd,
                                              student_lse=ls, teacher_lse=lt, sigma=sg,
                                              grad_student=grad, stream=stream, options=opts_alt)

    def vocab_shards():  # the vocabulary-parallel step with 2 shards on this GPU
        vocab_parallel.forward_backward_local(w.student, w.teacher, w.target, 2, w.grad_ce,
                                              w.grad_tvd, w.ignore_index, stream=stream)

    ce_lse = torch.empty_like(ce)
    signs = torch.empty(BT, binding.fused_ce_tvd_signs_row_bytes(V, w.student.dtype), device=dev,
                        dtype=torch.uint8)
    sign_bytes = BT * signs.shape[1]

    def fwd_signs():  # the forward that keeps sign words for its backward
        binding.fused_ce_tvd_forward_signs(w.student, w.teacher, w.target, w.ignore_index, ce=ce,
                                           tvd=tvd, student_lse=ls, teacher_lse=lt, sigma=sg,
                                           signs=signs, stream=stream, options=opts)

    def bwd_signs():
        binding.fused_ce_tvd_backward_signs(w.student, w.teacher, w.target, ls, lt, sg, signs,
                                            w.grad_ce, w.grad_tvd, w.ignore_index,
                                            grad_student=grad, stream=stream)

    def ce_fwd():  # the cross-entropy subset: student only
        binding.ce_forward(w.student, w.target, w.ignore_index, ce=ce, lse=ce_lse, stream=stream,
                           options=opts)

    def ce_bwd():
        binding.ce_backward(w.student, w.target, ce_lse, w.grad_ce, w.ignore_index,
                            grad_logits=grad, stream=stream)

    def ce_single():  # cross-entropy forward + backward in one launch
        binding.ce_forward_backward(w.student, w.target, w.grad_ce, w.ignore_index, ce=ce,
                                    lse=ce_lse, grad_logits=grad, stream=stream, options=opts)

    # the launches of one step of each path, with the algorithmic bytes of each launch
    paths = {
        "two": [("forward", fwd, 2 * BT * V * elem), ("backward", bwd, 3 * BT * V * elem)],
        "single": [("forward_backward", single, 3 * BT * V * elem)],
        "single_alt_ring": [("forward_backward_alt_ring", single_alt, 3 * BT * V * elem)],
        # vocabulary shards: passes 1 and 2 read both tensors, pass 3 reads both
        # and writes the gradient (7 V e per row), plus the merges
        "vocab2": [("vocab_parallel_2_shards", vocab_shards, 7 * BT * V * elem)],
        "ce": [("ce_forward", ce_fwd, BT * V * elem), ("ce_backward", ce_bwd, 2 * BT * V * elem)],
        "ce_single": [("ce_forward_backward", ce_single, 2 * BT * V * elem)],
        # two launches with sign words: the backward reads the student and the
        # bits (V/8 bytes per bf16 row) instead of the teacher
        "two_signs": [("forward_signs", fwd_signs, 2 * BT * V * elem + sign_bytes),
                      ("backward_signs", bwd_signs, 2 * BT * V * elem + sign_bytes)],
    }

    def time_path(name, K, sampler=None):
        launches = paths[name]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
              for _ in range(K)]
        if sampler:
            sampler.__enter__()
        barrier(world)
        torch.cuda.synchronize(dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            for i, (_, fn, _) in enumerate(launches):
                fn()
                ev[k][i + 1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        if sampler:
            sampler.__exit__(None, None, None)
        per = {}
        for i, (kname, _, nbytes) in enumerate(launches):
            kms = sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)) / K
            per[kname] = {"ms": kms, "gbs": nbytes / (kms * 1e-3) / 1e9, "bytes": nbytes}
        ms = sharding.max_over_ranks(start.elapsed_time(end) / K, world, dev)
        return ms, per

    for _ in range(args.warmup):
        for name in paths:
            for _, fn, _ in paths[name]:
                fn()
    torch.cuda.synchronize(dev)

    K = args.steps
    clocks = ClockSampler(local) if not args.no_clocks else None
    ms, kernels = time_path(args.path, K, clocks)
    value = world * BT / (ms * 1e-3)
    other_name = "two" if args.path == "single" else "single"
    other = None
    ce_path = None
    signs_path = None
    alt_ring_path = None
    vocab_path = None
    if not args.no_other:
        oms, okern = time_path(other_name, K)
        other = {"path": other_name, "ms_per_step": oms, "value": world * BT / (oms * 1e-3),
                 "kernels": okern}
        # cross-entropy alone (student logits only): forward + backward, 3 V e per row
        cms, ckern = time_path("ce", K)
        c1ms, c1kern = time_path("ce_single", K)
        ce_path = {"path": "ce", "ms_per_step": cms, "value": world * BT / (cms * 1e-3),
                   "unit": "tokens/s", "kernels": ckern,
                   "single_launch": {"ms_per_step": c1ms, "value": world * BT / (c1ms * 1e-3),
                                     "kernels": c1kern}}
        sms_, skern = time_path("two_signs", K)
        signs_path = {"path": "two_signs", "ms_per_step": sms_,
                      "value": world * BT / (sms_ * 1e-3), "unit": "tokens/s", "kernels": skern}
        vms, vkern = time_path("vocab2", max(1, K // 4))
        vocab_path = {"path": "vocab2", "shards": 2, "ms_per_step": vms,
                      "value": world * BT / (vms * 1e-3), "unit": "tokens/s", "kernels": vkern}
        ams, akern = time_path("single_alt_ring", K)
        alt_ring_path = {"path": "single", "ring": ("tma" if alt_ring == binding.RING_TMA
                                                    else "cp.async"),
                         "ms_per_step": ams, "value": world * BT / (ams * 1e-3),
                         "unit": "tokens/s", "kernels": akern}

    peaks = measured_peaks()
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    traffic = None
    if os.path.exists(PROFILE_SUMMARY):
        with open(PROFILE_SUMMARY) as f:
            prof = json.load(f)
        ent = prof.get("kernels", {}).get(dom)
        if (ent and prof.get("source_hash") == kernel_source_hash()
                and prof.get("workload") == args.workload):
            traffic = ent["bytes_per_launch_full"]
    # the metric's GB/s: bytes a step must move at minimum, over the step time
    step_bytes = sum(b for _, _, b in paths[args.path])
    step_gbs = step_bytes / (ms * 1e-3) / 1e9
    two_bytes = sum(b for _, _, b in paths["two"])

    # ---- end to end through the C ABI's host-buffer entry point: pinned host
    # logits, targets and upstream gradients in; the student gradient and the
    # five per-row outputs out, every step
    e2e = None
    if not args.no_e2e:
        hs = w.student.cpu().pin_memory()
        ht = w.teacher.cpu().pin_memory()
        htg = w.target.cpu().pin_memory()
        hgc = w.grad_ce.cpu().pin_memory()
        hgt = w.grad_tvd.cpu().pin_memory()
        houts = [torch.empty(BT, pin_memory=True) for _ in range(5)]
        hgrad = torch.empty(BT, V, dtype=w.student.dtype, pin_memory=True)
        hstatus = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        rows_e2e = min(args.e2e_block_rows, BT)
        wsp = torch.empty(binding.fused_ce_tvd_host_workspace_size(V, w.student.dtype, rows_e2e),
                          device=dev, dtype=torch.uint8)
        h2d = sum(x.numel() * x.element_size() for x in (hs, ht, htg, hgc, hgt))
        d2h = hgrad.numel() * hgrad.element_size() + 5 * BT * 4 + 4

        def e2e_step():
            binding.fused_ce_tvd_forward_backward_host(
                hs, ht, htg, hgc, hgt, w.ignore_index, ce=houts[0], tvd=houts[1],
                student_lse=houts[2], teacher_lse=houts[3], sigma=houts[4], grad_student=hgrad,
                block_rows=rows_e2e, workspace=wsp, status=hstatus, stream=stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        E = max(1, args.e2e_steps)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(E):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = sharding.max_over_ranks(a.elapsed_time(b) / E, world, dev)
        if int(hstatus.item()) != 0:
            raise RuntimeError(f"device status {int(hstatus.item())} in the end-to-end run")
        e2e = {"value": world * BT / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": E, "api": "fused_ce_tvd_forward_backward_host (C ABI, host buffers)",
               "block_rows": rows_e2e,
               "link_gbs": (h2d + d2h) / (e2e_ms * 1e-3) / 1e9}
        del hs, ht, hgrad, wsp

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.workload)

    if rank == 0:
        k = kernels[dom]
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "BT": BT, "V": V,
                       "logit_dtype": "bf16" if elem == 2 else "f32",
                       "path": args.path,
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "forward_ctas_per_row": args.cluster or "auto",
                       "ring": {0: "auto", 1: "cp.async", 2: "tma"}[args.ring],
                       "l2": "no flush: each step streams >= 7.4 GB, far above the 129 MB L2"
                       if args.rows is None else "reduced rows"},
            # GB/s of the bytes a step must move (3 V e per row in one launch) and the
            # same step time against the two-launch minimum (5 V e per row)
            "hbm_gbs": step_gbs,
            "hbm_frac": step_gbs / peaks["hbm_gbs"],
            "two_launch_equivalent_gbs": two_bytes / (ms * 1e-3) / 1e9,
            "kernels": kernels,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": k["gbs"],
                         "peak": peaks["hbm_gbs"], "peak_source": peaks["source"],
                         "unit": "GB/s", "frac": k["gbs"] / peaks["hbm_gbs"],
                         "traffic": traffic},
            "gpu_launches": len(paths[args.path]) * K,
            "other_path": other,
            "ce_path": ce_path,
            "signs_path": signs_path,
            "alt_ring_path": alt_ring_path,
            "vocab_path": vocab_path,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks.summary() if clocks else None,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
