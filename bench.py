#!/usr/bin/env python
"""Benchmark of the fused linear cross-entropy (forward + backward) on GB300.

One step = flce_forward + flce_backward over one batch of the Qwen3-8B-like head
(N=16384 tokens, D=4096, V=151936, bf16, mean reduction) -- the workload the
headline metric is quoted on.  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload qwen8b]
    python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream,
max over ranks.  The inputs of every benchmark head but the tiny one are larger
than L2 (the Qwen3-8B-like head alone is ten times the 129 MB L2), so no flush
is needed between their steps; smaller inputs get a 256 MB buffer written
between steps, outside the steps' events.  For N > 1 every rank runs its own
replica of the workload (independent batches; the loss needs no exchange), so
scaling is weak.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd tokens/s and TFLOP/s (% of GB300 bf16 tensor peak)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# ----------------------------------------------------------------------------- utilities
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["flce", "reference"], default="flce")
    ap.add_argument("--workload", default="qwen8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle sample rows (0 = automatic)")
    ap.add_argument("--tokens", type=int, default=0, help="override N (profiling captures of a small case)")
    ap.add_argument("--vocab", type=int, default=0, help="override V (profiling captures of a small case)")
    ap.add_argument("--hidden", type=int, default=0, help="override D (calibration sweeps)")
    ap.add_argument("--separate", action="store_true",
                    help="flce_forward + flce_backward per step instead of one flce_forward_backward call")
    ap.add_argument("--autograd", action="store_true",
                    help="time the torch autograd wrapper: linear_cross_entropy(...) + loss.backward() per step "
                         "(gradients computed in the forward for mean / sum); no e2e leg")
    ap.add_argument("--grad-in-backward", action="store_true",
                    help="with --autograd: the separate backward instead of gradients in the forward")
    ap.add_argument("--bwd", default="auto", choices=["auto", "recompute", "keep_logits"],
                    help="backward algorithm of the fused call (FLCE_FLAG_BWD_*); auto keeps the logits of "
                         "token chunks from D = 1152 up")
    ap.add_argument("--compact", action="store_true",
                    help="gather the valid tokens first (FLCE_FLAG_COMPACT_VALID)")
    ap.add_argument("--token-chunk", type=int, default=0,
                    help="rows per token chunk of the keep-logits backward (0 = automatic; tuning)")
    ap.add_argument("--gemm-mode", type=int, default=0, choices=[0, 1, 2],
                    help="GEMM kernel: 0 automatic, 1 single CTA, 2 CTA pair (A/B timing)")
    ap.add_argument("--e2e-grads", action="store_true",
                    help="the e2e leg also reads dhidden, dweight and dbias back to pinned host memory every step "
                         "(by default only the loss and the metrics return; the gradients stay on the device)")
    ap.add_argument("--valid-frac", type=float, default=0.0,
                    help="prompt-completion batches: only the last fraction of every 2048-token sequence has a "
                         "target (the prompt before it is ignored); 0 keeps the workload's own ignore pattern")
    ap.add_argument("--frozen-head", action="store_true",
                    help="the head and bias are not trained (FLCE_FLAG_FROZEN_HEAD, as in LoRA training): the "
                         "backward forms dhidden only")
    ap.add_argument("--dh-ksplit", type=int, default=0,
                    help="force the K splits of the recompute backward's dh product (0 = automatic; tuning)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Max of a scalar over all ranks (timing only; no data-path exchange)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.proc = None
        self.out = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(index)], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample_step(h_rows, W, b, t_rows, dloss, w):
    """One oracle forward + backward over a sample of tokens (the oracle as it stands)."""
    import oracle
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    f = oracle.forward(h_rows, W, b, t_rows, **kw)
    g = oracle.backward(h_rows, W, b, t_rows, dloss=dloss, **kw)
    return f, g


def cpu_inputs(w, rows):
    """The workload's tensors restricted to a token sample, on the CPU."""
    import torch

    from linear_cross_entropy_tmem_gb300.synthetic import make_inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    sample = w.scaled(n_tokens=max(rows, 1))
    h, W, b, t, dloss = make_inputs(sample, dev)
    out = [x.cpu() if x is not None else None for x in (h, W, b, t, dloss)]
    del h, W, b, t, dloss
    if dev == "cuda":
        torch.cuda.empty_cache()
    return out


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(w, rows=0, budget_s=15.0):
    """Time the oracle on a bounded sample of the workload (tokens/s on host cores)."""
    rows = rows or 32
    h, W, b, t, dloss = cpu_inputs(w, rows)
    t0 = time.perf_counter()
    oracle_sample_step(h, W, b, t, dloss, w)
    dt = time.perf_counter() - t0
    reps = 1
    while dt * (reps + 1) / reps < budget_s and dt < budget_s / 2 and reps < 4:
        t1 = time.perf_counter()
        oracle_sample_step(h, W, b, t, dloss, w)
        dt += time.perf_counter() - t1
        reps += 1
    value = rows * reps / dt
    return {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{rows} tokens x {reps} runs of the fp64 oracle forward+backward at full V={w.vocab}, "
                      f"D={w.hidden} ({dt:.1f} s)"}


def reference_arm(args):
    from linear_cross_entropy_tmem_gb300.synthetic import WORKLOADS
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = pick_workload(args)
    rows = args.cpu_rows or 16
    h, W, b, t, dloss = cpu_inputs(w, rows)
    for _ in range(args.warmup):
        oracle_sample_step(h, W, b, t, dloss, w)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(h, W, b, t, dloss, w)
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "n_tokens": w.n_tokens, "hidden": w.hidden, "vocab": w.vocab,
                   "sample_tokens_per_step": rows, "l2": "n/a (host)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{rows} tokens per step at full V and D, fp64 oracle forward+backward"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
class Runner:
    """Preallocated buffers and raw C-ABI calls for one forward + backward step."""

    def __init__(self, w, device, seed_offset=0, compact=False, fused=False, bwd="auto", autograd=False,
                 grad_in_forward=True, frozen_head=False, valid_frac=0.0):
        import torch

        import linear_cross_entropy_tmem_gb300.api as api
        from linear_cross_entropy_tmem_gb300 import binding as B
        from linear_cross_entropy_tmem_gb300.synthetic import make_inputs
        self.B = B
        self.lib = B.load()
        self.w = w
        self.device = device
        self.h, self.W, self.b, self.t, self.dloss = make_inputs(w.scaled(seed=w.seed + seed_offset), device)
        N, D, V = w.n_tokens, w.hidden, w.vocab
        if valid_frac > 0.0:  # prompt-completion batches: each 2048-token sequence's prompt is ignored
            pos = torch.arange(N, device=device) % 2048
            self.t[pos < round((1.0 - valid_frac) * 2048)] = -100
        self.prob = api.make_problem(N, D, V, hidden_dtype=self.h.dtype, bias_dtype=torch.bfloat16,
                                     logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction,
                                     compact=compact, bwd=bwd, frozen_head=frozen_head)
        f32 = dict(dtype=torch.float32, device=device)
        self.loss = torch.empty(N if w.reduction == "none" else 1, **f32)
        self.lse = torch.empty(N, **f32)
        self.correct = torch.empty(1, dtype=torch.int64, device=device)
        self.n_valid = torch.empty(1, dtype=torch.int64, device=device)
        self.ent_sum = torch.empty(1, **f32)
        self.dh = torch.empty_like(self.h)
        self.frozen_head = frozen_head  # dhidden only: no dweight / dbias buffers are passed
        self.dW = torch.empty_like(self.W) if not frozen_head else None
        self.db = torch.empty_like(self.b) if self.b is not None and not frozen_head else None
        self.ws_f = torch.empty(api.flce_workspace_size(self.prob, False), dtype=torch.uint8, device=device)
        self.ws_b = torch.empty(api.flce_workspace_size(self.prob, True), dtype=torch.uint8, device=device)
        self.fused = fused
        self.ws_fb = torch.empty(api.flce_workspace_size(self.prob, 2) if fused else 256, dtype=torch.uint8,
                                 device=device)
        self.stream = torch.cuda.current_stream(device)
        p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
        s = ctypes.c_void_p(self.stream.cuda_stream)
        self.fwd_args = (ctypes.byref(self.prob), p(self.h), p(self.W), p(self.b), p(self.t), p(self.loss),
                         p(self.lse), None, p(self.correct), p(self.n_valid), p(self.ent_sum), p(self.ws_f),
                         self.ws_f.numel(), s)
        self.bwd_args = (ctypes.byref(self.prob), p(self.h), p(self.W), p(self.b), p(self.t), p(self.lse),
                         p(self.n_valid), p(self.dloss), p(self.dh), p(self.dW), p(self.db), p(self.ws_b),
                         self.ws_b.numel(), s)

        self.autograd = autograd
        self.grad_in_forward = grad_in_forward
        if autograd:  # a frozen head: the weight and bias leaves do not require gradients
            self.leaves = [x.detach().requires_grad_(i == 0 or not frozen_head) if x is not None else None
                           for i, x in enumerate((self.h, self.W, self.b))]
        self.fb_args = (ctypes.byref(self.prob), p(self.h), p(self.W), p(self.b), p(self.t), p(self.dloss),
                        p(self.loss), p(self.lse), None, p(self.correct), p(self.n_valid), p(self.ent_sum),
                        p(self.dh), p(self.dW), p(self.db), p(self.ws_fb), self.ws_fb.numel(), s)

    def step(self):
        if self.autograd:  # the torch API a training loop calls
            import linear_cross_entropy_tmem_gb300 as F
            h, W, b = self.leaves
            for x in self.leaves:
                if x is not None:
                    x.grad = None
            w = self.w
            loss = F.linear_cross_entropy(h, W, self.t, b, logit_scale=w.logit_scale, softcap=w.softcap,
                                          reduction=w.reduction, grad_in_forward=self.grad_in_forward)[0]
            loss.backward(self.dloss if w.reduction == "none" else None)
            return
        if self.fused:
            self.B.check(self.lib.flce_forward_backward(*self.fb_args), "flce_forward_backward")
            return
        self.B.check(self.lib.flce_forward(*self.fwd_args), "flce_forward")
        self.B.check(self.lib.flce_backward(*self.bwd_args), "flce_backward")

    def input_bytes(self):
        return sum(x.numel() * x.element_size() for x in (self.h, self.W, self.b, self.t, self.dloss) if x is not None)


def kernel_source_hash():
    """Hash of the kernel sources with comments and whitespace removed, so that documentation edits
    keep committed counters valid while any code change invalidates them."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_cross_entropy_tmem_gb300", "csrc")
    strip = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            code = "".join(strip.sub("", fh.read()).split())
        h.update(f.encode())
        h.update(code.encode())
    return h.hexdigest()[:16]


def committed_traffic(kind, workload, backward):
    """DRAM bytes per launch from the committed ncu summary (workload -> backward algorithm ->
    launch kind), if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    e = rec.get(workload, {}).get(backward, {}).get(kind)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def kernel_model(w, keep, rows, launches, h_terms, grad_h_terms):
    """Algorithmic work of each launch kind over one step: flops (2 per multiply-add of the
    product) and the bytes the kind must read and write to do its part (operands read, results
    written), counting the re-reads and accumulator traffic that the chosen algorithm itself
    implies.  Returns {kind: (flops, bytes read, bytes written)}.

    rows: tokens the products run over; launches: {kind: launches per step}; h_terms: bf16 terms the
    logit products read of the hidden state (1 for bf16, 2 or 3 for fp32); grad_h_terms: those the
    dW product reads.  Kept logits run per token chunk (W read once per chunk; dW accumulated in
    fp32 across chunks); the recompute runs per vocabulary chunk (h read once per chunk)."""
    R, V, D = float(rows), float(w.vocab), float(w.hidden)
    eh = 4.0 if w.hidden_dtype.itemsize == 4 else 2.0
    out = {}
    prod = 2.0 * R * V * D
    if keep:
        nc = max(1, launches.get("bwd_logit_grad", 1))
        out["fwd_logits"] = (prod, 2 * h_terms * R * D + 2 * nc * V * D, 4 * R * V)
        out["bwd_logit_grad"] = (0.0, 4 * R * V, 2 * R * V)
        out["bwd_dhidden"] = (prod, 2 * R * V + 2 * nc * V * D, eh * R * D)
        out["bwd_dweight"] = (prod, 2 * R * V + 2 * grad_h_terms * R * D + 4 * V * D * (nc - 1),
                              4 * V * D * (nc - 1) + 2 * V * D)
    else:
        nv = max(1, launches.get("bwd_recompute", 1))
        out["fwd_logits"] = (prod, 2 * h_terms * R * D + 2 * V * D, 0.0)
        out["bwd_recompute"] = (prod, 2 * nv * h_terms * R * D + 2 * V * D, 2 * R * V)
        out["bwd_dweight"] = (prod, 2 * R * V + 2 * nv * grad_h_terms * R * D, 2 * V * D)
        out["bwd_dhidden"] = (prod, 2 * R * V + 2 * V * D + 4 * R * D * (nv - 1), 4 * R * D * (nv - 1) + eh * R * D)
    return out


def write_bandwidth(device):
    """Pure HBM write bandwidth measured live: best of 5 memsets of 1 GiB (GB/s).  On GB300 it is
    well below the copy bandwidth (writes alone do not reach the read + write rate of a copy), so
    the floor of a kernel that mostly writes is its written bytes at this rate."""
    import torch
    x = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    for _ in range(3):
        x.zero_()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        x.zero_()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    del x
    return (1 << 30) / (best * 1e-3) / 1e9


def pick_workload(args):
    from linear_cross_entropy_tmem_gb300.synthetic import WORKLOADS
    w = WORKLOADS[args.workload]
    kw = {}
    if args.tokens:
        kw["n_tokens"] = args.tokens
    if args.vocab:
        kw["vocab"] = args.vocab
    if args.hidden:
        kw["hidden"] = args.hidden
    if kw:
        w = w.scaled(name=f"{w.name} (N={kw.get('n_tokens', w.n_tokens)}, D={kw.get('hidden', w.hidden)}, "
                          f"V={kw.get('vocab', w.vocab)})", **kw)
    return w


def flce_arm(args):
    import torch

    from linear_cross_entropy_tmem_gb300 import binding as B
    from linear_cross_entropy_tmem_gb300.synthetic import WORKLOADS
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist("nccl")
    w = pick_workload(args)
    lib = B.load()
    B.check(lib.flce_testing_set_gemm_mode(args.gemm_mode), "gemm mode")
    B.check(lib.flce_testing_set_tuning(0, args.dh_ksplit), "dh K splits")
    B.check(lib.flce_testing_set_token_chunk(args.token_chunk), "token chunk")  # before sizing the workspace
    run = Runner(w, device, seed_offset=rank, compact=args.compact, fused=not args.separate, bwd=args.bwd,
                 autograd=args.autograd, grad_in_forward=not args.grad_in_backward, frozen_head=args.frozen_head,
                 valid_frac=args.valid_frac)
    if args.autograd:
        if args.compact:
            raise SystemExit("--autograd does not combine with --compact")
        args.no_e2e = True

    for _ in range(args.warmup):
        run.step()
    torch.cuda.synchronize()

    # ---- device-timed region, with the launch log bracketing every kernel
    n_launch_per_step = 128
    cap = n_launch_per_step * args.steps
    recs = (B.FlceLaunchRecord * cap)()
    events = []
    for i in range(cap):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()  # torch creates the CUDA event on its first record
        e1.record()
        events.append((e0, e1))
        recs[i].begin_event = ctypes.c_void_p(e0.cuda_event)
        recs[i].end_event = ctypes.c_void_p(e1.cuda_event)
    count = ctypes.c_int32(0)
    # Operands that fit in L2 (129 MB) would stay there from one step to the next: write a 256 MB
    # buffer between steps instead, outside the steps' events.
    l2_bytes = 129 << 20
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device) if run.input_bytes() < 2 * l2_bytes else None
    clocks = ClockSampler(local)
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    launches0 = lib.flce_testing_launch_count()
    B.check(lib.flce_testing_set_launch_log(recs, cap, ctypes.byref(count)), "launch log")
    step_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    step_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    start.record()
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(k & 0xFF)  # evict the previous step's operands from L2 (outside the step's events)
        step_starts[k].record()
        run.step()
        step_ends[k].record()
    end.record()
    torch.cuda.synchronize()
    B.check(lib.flce_testing_set_launch_log(None, 0, None), "launch log")
    launches = lib.flce_testing_launch_count() - launches0
    barrier(dist, device)
    clock = clocks.stop()
    per_step = [step_starts[k].elapsed_time(step_ends[k]) for k in range(args.steps)]
    # back to back: the whole region; with an L2 flush between steps: the steps alone
    ms = start.elapsed_time(end) / args.steps if flush is None else sum(per_step) / args.steps
    qs = statistics.quantiles(per_step, n=10, method="inclusive") if len(per_step) > 1 else per_step * 9
    step_quantiles = {"p20": qs[1], "p50": statistics.median(per_step), "p80": qs[7], "min": min(per_step),
                      "max": max(per_step)}
    status = ctypes.c_int(0)
    if not args.autograd:  # (the autograd API allocates its workspace per call)
        ws_status = run.ws_fb if run.fused else run.ws_b
        B.check(lib.flce_read_device_status(ctypes.c_void_p(ws_status.data_ptr()), None, ctypes.byref(status)),
                "status")
        if status.value != 0:
            raise RuntimeError(f"device status {status.value} during the timed region")

    # The events that bracket every launch above also serialise the launches: the GEMMs, launched
    # as programmatic dependents, cannot overlap their set-up with the previous kernel's end there.
    # The same K steps again with events around whole steps only show what that costs (a few us
    # per launch: visible on small heads, negligible on the large ones).
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(k & 0xFF)
        step_starts[k].record()
        run.step()
        step_ends[k].record()
    torch.cuda.synchronize()
    clean = [step_starts[k].elapsed_time(step_ends[k]) for k in range(args.steps)]
    step_clean = {"p50": statistics.median(clean), "mean": sum(clean) / len(clean),
                  "note": "the same K steps again, without the per-launch events of the timed region"}

    per_kind = {}
    for i in range(count.value):
        k = B.LAUNCH_KINDS[recs[i].kind]
        d = per_kind.setdefault(k, [0, 0.0])
        d[0] += 1
        d[1] += events[i][0].elapsed_time(events[i][1])
    # Tokens the products run over: all of them, or the valid ones under compaction.
    rows_mult = int(run.n_valid.item()) if args.compact else w.n_tokens
    keep = "bwd_logit_grad" in per_kind  # the token-chunked backward ran (6NVD instead of 8NVD)
    h_terms = 1 if w.hidden_dtype == torch.bfloat16 else 2
    model = kernel_model(w, keep, rows_mult, {k: v[0] // args.steps for k, v in per_kind.items()}, h_terms, 1)
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    write_gbs = write_bandwidth(device)
    # a kernel inside a timed region of half a second or more runs under the sustained power cap
    timed_s = ms * args.steps * 1e-3
    peak_f, peak_f_kind = (peak_sus, "sustained") if timed_s >= 0.5 else (peak_burst, "burst")
    kernels = {}
    for k, (n_l, t_ms) in sorted(per_kind.items()):
        e = {"launches": n_l, "ms_per_step": t_ms / args.steps}
        if k in model:
            fl, rd, wr = model[k]
            t_s = t_ms * 1e-3 / args.steps
            floors = {"tensor": fl / (peak_f * 1e12), "hbm": (rd + wr) / (peak_bw * 1e9),
                      "hbm_write": wr / (write_gbs * 1e9)}
            limit = max(floors, key=floors.get)
            tensor = limit == "tensor"
            e.update({"flops_per_step": fl, "bytes_per_step": rd + wr, "bytes_written_per_step": wr,
                      "tflops": fl / t_s / 1e12 if fl else None, "gbs": (rd + wr) / t_s / 1e9,
                      "bound": "tensor" if tensor else "hbm",
                      "frac": (fl / t_s / 1e12 / peak_f) if tensor else ((rd + wr) / t_s / 1e9 / peak_bw),
                      "floor": limit, "frac_of_floor": floors[limit] / t_s})
        kernels[k] = e
    dominant = max(model, key=lambda k: per_kind.get(k, [0, 0.0])[1])
    dk = kernels[dominant]
    n_l, t_ms = per_kind[dominant]
    if dk["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dk["tflops"], "peak": peak_f, "unit": "TFLOP/s",
                "peak_kind": f"bf16 {peak_f_kind} ({peak_src})"}
    else:
        roof = {"bound": "hbm", "achieved": dk["gbs"], "peak": peak_bw, "unit": "GB/s",
                "peak_kind": f"HBM copy bandwidth ({peak_src})"}
    roof.update({"kernel": dominant, "frac": roof["achieved"] / roof["peak"],
                 "flops_per_launch": model[dominant][0] / max(1, n_l // args.steps),
                 "bytes_per_launch": (model[dominant][1] + model[dominant][2]) / max(1, n_l // args.steps),
                 "launches": n_l, "avg_launch_ms": t_ms / n_l,
                 # the largest of the tensor, HBM and HBM-write floors, over the measured time
                 "floor": dk["floor"], "frac_of_floor": dk["frac_of_floor"],
                 "hbm_write_gbs_measured": write_gbs})

    ms_max = max_over_ranks(dist, ms, device)
    tokens = w.n_tokens * world
    value = tokens / (ms_max * 1e-3)
    tflops = w.flops() * world / (ms_max * 1e-3) / 1e12
    # executed products: 6NVD with kept logits, 8NVD with the recompute, 2NVD fewer with a frozen head
    exec_flops = 8.0 * rows_mult * w.vocab * w.hidden * ((0.75 if keep else 1.0) - (0.25 if args.frozen_head else 0.0))
    tflops_exec = exec_flops * world / (ms_max * 1e-3) / 1e12

    # ---- end to end through host buffers: H2D inputs, step, D2H loss + metrics
    e2e = None
    if not args.no_e2e:
        # End to end through host buffers: every step copies its inputs from pinned host memory
        # and reads its scalar results back.  Two device buffer sets alternate, so that the
        # copy of step k+1's inputs (copy stream) runs during step k's compute, as a training
        # loop that prefetches its next batch would.
        runs = [run, Runner(w, device, seed_offset=rank, compact=args.compact, fused=not args.separate,
                            bwd=args.bwd, frozen_head=args.frozen_head, valid_frac=args.valid_frac)]
        host = {k: getattr(run, k).to("cpu").pin_memory() for k in ("h", "W", "t", "dloss")
                if getattr(run, k) is not None}
        if run.b is not None:
            host["b"] = run.b.to("cpu").pin_memory()
        out_host = [torch.empty(4, dtype=torch.float64).pin_memory() for _ in range(2)]
        res = [torch.empty(4, dtype=torch.float64, device=device) for _ in range(2)]
        main = torch.cuda.current_stream(device)
        copy_stream = torch.cuda.Stream(device)
        copied = [torch.cuda.Event() for _ in range(2)]
        released = [torch.cuda.Event() for _ in range(2)]  # the step that last used buffer set i is done
        grads = [n for n in ("dh", "dW", "db") if getattr(run, n) is not None] if args.e2e_grads else []
        grads_host = [{n: torch.empty(getattr(run, n).shape, dtype=getattr(run, n).dtype).pin_memory()
                       for n in grads} for _ in range(2)]
        d2h_stream = torch.cuda.Stream(device) if grads else None
        d2h_done = [torch.cuda.Event() for _ in range(2)]  # buffer set i's gradients have reached the host

        def e2e_step(k):
            i = k % 2
            r = runs[i]
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(released[i])
                for name, v in host.items():
                    getattr(r, name).copy_(v, non_blocking=True)
                copied[i].record(copy_stream)
            main.wait_event(copied[i])
            if grads:
                main.wait_event(d2h_done[i])  # step k-2's gradients have left this buffer set
            r.step()
            res[i][0] = r.loss[0]
            res[i][1] = r.correct[0]
            res[i][2] = r.n_valid[0]
            res[i][3] = r.ent_sum[0]
            out_host[i].copy_(res[i], non_blocking=True)
            released[i].record(main)
            if grads:  # read the gradients back on a third stream, during the next step
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(released[i])
                    for n in grads:
                        grads_host[i][n].copy_(getattr(r, n), non_blocking=True)
                    d2h_done[i].record(d2h_stream)

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize()
        barrier(dist, device)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        copy_stream.wait_stream(main)  # the first copy starts inside the timed region
        for k in range(args.steps):
            e2e_step(k)
        for ev in d2h_done if grads else ():
            main.wait_event(ev)  # the last gradients are on the host
        s1.record()  # after the last step, which waited for its copies, and its result copy
        torch.cuda.synchronize()
        e_ms = max_over_ranks(dist, s0.elapsed_time(s1) / args.steps, device)
        d2h = out_host[0].numel() * out_host[0].element_size() + sum(
            v.numel() * v.element_size() for v in grads_host[0].values())
        e2e = {"value": tokens / (e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(sum(v.numel() * v.element_size() for v in host.values())),
               "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms,
               "returns": ("loss, correct, n_valid, entropy_sum and the gradients dhidden, dweight"
                           + (", dbias" if "db" in grads else "") if grads else
                           "loss, correct, n_valid and entropy_sum (32 bytes); dhidden and dweight stay on the "
                           "device, where an optimizer step would use them"),
               "overlap": "step k+1's inputs are copied on a second stream during step k (two device buffer sets)"
                          + ("; step k's gradients are read back on a third stream during step k+1" if grads
                             else "")}
        del runs

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_rows)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "ms_per_step_quantiles": step_quantiles,
            "ms_per_step_without_launch_events": step_clean,
            "vs_baseline": None, "dtype": "bf16" if w.hidden_dtype == torch.bfloat16 else "f32+bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "n_tokens": w.n_tokens, "hidden": w.hidden, "vocab": w.vocab,
                       "reduction": w.reduction, "parallelism": f"replicas x{world}" if world > 1 else "none",
                       "gemm_mode": ["auto", "single-cta", "cta-pair"][args.gemm_mode],
                       "compact_valid_tokens": bool(args.compact),
                       "valid_tokens": None if args.autograd else int(run.n_valid.item()),
                       "entry": ("linear_cross_entropy + backward (autograd, gradients "
                                 + ("in the backward)" if args.grad_in_backward else "in the forward)"))
                       if args.autograd else
                       "flce_forward + flce_backward" if args.separate else "flce_forward_backward",
                       "backward": (("keep_logits (token chunks, 4NVD: frozen head, dhidden only)" if keep else
                                     "recompute (6NVD: frozen head, dhidden only)") if args.frozen_head else
                                    "keep_logits (token chunks, 6NVD)" if keep else "recompute (8NVD)"),
                       "l2": ("inputs larger than L2 (129 MB), no flush" if flush is None else
                              "256 MB buffer written between steps (outside the steps' events) to flush L2")},
            # executed flops: 6NVD with kept logits, 8NVD with the recompute; the metric's own
            # accounting counts 8NVD per forward + backward whatever the algorithm
            "tflops": tflops_exec,
            "tflops_8nvd_accounting": tflops,
            "flops_per_step": {"executed": exec_flops, "metric_8nvd": w.flops()},
            "pct_of_peak": {"of_burst": tflops_exec / peak_burst, "of_sustained": tflops_exec / peak_sus,
                            "source": peak_src, "flops": "executed"},
            "roofline": dict(roof, traffic=committed_traffic(dominant, args.workload,
                                                             "keep_logits" if keep else "recompute")
                             if not (args.tokens or args.vocab or args.hidden or args.compact) else None),
            "kernels": kernels,
            "gpu_launches": int(launches),
            "clocks": clock,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return reference_arm(args)
    return flce_arm(args)


if __name__ == "__main__":
    sys.exit(main())
