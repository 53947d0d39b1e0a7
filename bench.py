#!/usr/bin/env python3
"""Benchmark of the fused LM-head projection + cross-entropy, forward + backward.

Metric: credited TFLOP/s counting 6*N*H*V per step (2NHV for the logits, 2NHV
each for dX and dW), with the extra device memory the op needs beside it.
A step is one flce_fwd_bwd over one synthetic batch (loss, lse, dX, dW) on the
bounded, V-independent workspace (logits recomputed in the backward pass:
8NHV executed, 6NHV credited).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload n131072_h4096_v131072]
                    [--path bounded|rowchunk] [--impl flce|reference]

Default workload: the 128K-token x 128K-vocabulary case (N = 131072, H = 4096,
V = 131072, uniform labels with 3% ignore_index, mean reduction), whose bf16
logits would take 32 GiB.  The line also carries the row-chunk path
(flce_fwd_bwd_rowchunk, 6NHV executed, a workspace that grows with V) on the
same inputs, and both paths on the three other benchmark workloads
(``workloads``), each measured with the same timing discipline.
Under torchrun each rank runs its own batch of that shape on its own GPU
(weak scaling, no collective on the data path); rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead (bounded
row samples of the same workload), the deliberately slow definition the
CUDA path is checked against.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused linear-CE fwd+bwd TFLOP/s (6NHV), % of BF16 tensor peak; extra HBM"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 512 << 20


HEADLINE = "n131072_h4096_v131072"
OTHER_WORKLOADS = ("n8192_h2048_v32000", "n8192_h4096_v128256", "n32768_h4096_v151936")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, help="one of synth.WORKLOADS")
    ap.add_argument("--path", choices=["bounded", "rowchunk"], default="bounded",
                    help="bounded: flce_fwd_bwd, V-independent workspace (8NHV executed); rowchunk: "
                         "flce_fwd_bwd_rowchunk, logits computed once (6NHV), workspace grows with V")
    ap.add_argument("--impl", choices=["flce", "reference"], default="flce")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-naive", action="store_true", help="skip timing the unfused torch lm_head + cross_entropy")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other path and the other workloads (the 'rowchunk' and 'workloads' keys)")
    ap.add_argument("--other-steps", type=int, default=10, help="timed steps of each other path / workload")
    ap.add_argument("--op", choices=["fwd_bwd", "topk", "soft"], default="fwd_bwd",
                    help="fwd_bwd: fused loss + gradients (the benchmark); topk: per-row top-k logits; "
                         "soft: KL against sparse soft targets, forward + backward")
    ap.add_argument("--k", type=int, default=8, help="k of --op topk / soft")
    ap.add_argument("--reduction", choices=["mean", "sum", "none"], default=None, help="override the workload's")
    ap.add_argument("--shift", type=int, default=0, help="1: causal next-token shift inside the kernels")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_config(name, problem_kw, l2_note, world):
    import synth
    c = synth.WORKLOADS[name]
    return {
        "workload": f"{name}: {c['name']}",
        "n_tokens_per_rank": c["n"], "hidden": c["h"], "vocab": c["v"],
        "labels": c["labels"] + ("(s=1.1)" if c["labels"] == "zipf" else ""),
        "ignore_frac": c["ignore_frac"], "reduction": c["reduction"],
        "x_std": c["x_std"], "w_std": c["w_std"], "outlier_rows": c.get("outlier_rows", 0),
        "l2": l2_note,
        "parallelism": f"replicas x{world} (rows sharded by rank, no collective)" if world > 1 else "single GPU",
    }


def arm_config(args, world):
    """The `config` of the benchmark line, the same for both arms."""
    return dict(workload_config(args.workload, None, f"inputs larger than L2, and a {L2_FLUSH_BYTES >> 20} MiB write "
                                "between steps (outside the per-step events)", world), path=args.path)


def credited_flops(n, h, v):
    return 6.0 * n * h * v


def rank_seed(base_seed, rank):
    """Each rank draws its own batch of the workload's shape (rows shard by rank)."""
    return base_seed + 1000 * rank


def max_over_ranks(value, dist, device):
    """The slowest rank's time decides the whole job's time."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank_step, steps, max_ms):
    """Whole-job throughput: every rank's credited flops over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_ms / 1e3) / 1e12


# ----------------------------------------------------------------------------- CPU oracle timing

def oracle_sample_seconds(problem, rows, Wd=None):
    """Time the fp64 oracle (loss, lse, dX, dW) on the first `rows` rows with the full W
    (``Wd``: W already widened to fp64, to reuse across samples)."""
    import oracle
    X = oracle.widen_bf16(problem.X[:rows])
    W = oracle.widen_bf16(problem.W) if Wd is None else Wd
    lab = problem.labels[:rows]
    t0 = time.perf_counter()
    oracle.full(X, W, lab, problem.ignore_index, problem.reduction)
    return time.perf_counter() - t0


def calibrate_rows(problem, target_s, max_rows, Wd=None):
    r = min(64, max_rows)
    dt = oracle_sample_seconds(problem, r, Wd)
    per_row = dt / r
    return int(max(1, min(max_rows, target_s / max(per_row, 1e-9))))


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def torch_naive(X, W, y, problem, flush, stream, torch, steps=5):
    """The unfused computation the fused call replaces, in plain torch: logits = X W^T (bf16),
    cross_entropy on their fp32 copy, autograd backward.  Time per step and the peak memory it
    allocates beyond its inputs, or the allocation failure."""
    import torch.nn.functional as F
    yl = y.long()

    def step():
        Xr = X.detach().requires_grad_()
        Wr = W.detach().requires_grad_()
        loss = F.cross_entropy((Xr @ Wr.T).float(), yl, ignore_index=problem.ignore_index,
                               reduction=problem.reduction)
        loss.backward()
        return loss

    dev = X.device
    need = 16 * problem.n * problem.v  # bf16 logits, their fp32 copy, fp32 log-softmax and its gradient, bf16 grad
    total = torch.cuda.get_device_properties(dev).total_memory
    if need > total // 2:
        return {"unavailable": f"needs about {need / 1e9:.0f} GB of device memory for [N,V] buffers "
                               f"(more than half of {total / 1e9:.0f} GB); not run"}
    try:
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        step()
        torch.cuda.synchronize()
        peak = torch.cuda.max_memory_allocated(dev) - base
        step()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
        ms = []
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[2 * i].record(stream)
            step()
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
        t = statistics.median(ms)
        return {"ms_per_step": t, "value": credited_flops(problem.n, problem.h, problem.v) / (t / 1e3) / 1e12,
                "unit": UNIT, "peak_alloc_delta_bytes": int(peak),
                "note": "torch: (X @ W.T).float() -> F.cross_entropy -> backward (cuBLAS + torch kernels), "
                        "median of 5 steps, L2 flushed between steps"}
    except torch.cuda.OutOfMemoryError as e:
        torch.cuda.empty_cache()
        return {"unavailable": f"out of device memory: {str(e).splitlines()[0][:160]}"}


def cpu_baseline(problem, target_s):
    import oracle
    Wd = oracle.widen_bf16(problem.W)
    rows = calibrate_rows(problem, target_s, problem.n, Wd)
    dt = oracle_sample_seconds(problem, rows, Wd)
    val = credited_flops(rows, problem.h, problem.v) / dt / 1e12
    return {"value": val, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 numpy oracle (loss, lse, dX, dW) on the first {rows} of {problem.n} rows with the full "
                      f"W [{problem.v}x{problem.h}], {dt:.1f} s; credited 6*rows*H*V flops; BLAS threads = numpy default"}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    import synth
    problem = synth.workload_problem(args.workload)
    Wd = oracle.widen_bf16(problem.W)
    total_steps = args.steps + args.warmup
    per_step_s = max(0.5, min(10.0, 120.0 / max(1, total_steps)))
    rows = calibrate_rows(problem, per_step_s, problem.n, Wd)
    for _ in range(args.warmup):
        oracle_sample_seconds(problem, rows, Wd)
    times = [oracle_sample_seconds(problem, rows, Wd) for _ in range(args.steps)]
    t = sum(times)
    val = credited_flops(rows, problem.h, problem.v) * args.steps / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": arm_config(args, world),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: fp64 numpy oracle (loss, lse, dX, dW) on the first {rows} of "
                                   f"{problem.n} rows with the full W"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock, throttle reasons and power every 20 ms,
    kept only when their timestamp falls inside the marked (timed) region."""
    # power.draw.instant: the power-capping decisions follow the instantaneous draw, which on
    # a heavy tensor-core load passes the limit within ~100 ms while the averaged draw lags
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.draw.instant")
    PERIOD_MS = 20

    def __init__(self, gpu_index):
        # nvidia-smi numbers every GPU of the machine; CUDA may see a subset
        # (CUDA_VISIBLE_DEVICES), so the GPU is named by its PCI bus id
        self.gpu = gpu_index
        try:
            import torch
            pr = torch.cuda.get_device_properties(gpu_index)
            self.gpu = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        except (ImportError, AttributeError, RuntimeError, AssertionError):
            pass
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows, total = [], 0
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 11:
                    continue
                total += 1
                when = self._when(parts[0])
                if self.t0 is not None and (when is None or when < self.t0 or (self.t1 and when > self.t1)):
                    continue
                rows.append(parts[1:])
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"], "samples": 0,
                    "samples_total": total}
        num = lambda x: x.replace(".", "").isdigit()  # noqa: E731
        sm = [float(r[1]) for r in rows if num(r[1])]
        smax = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        power = [float(r[9]) for r in rows if num(r[9])]
        capped = sum(1 for r in rows if r[8].lower().startswith("active"))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "sm_mhz_min": min(sm) if sm else None, "reasons": reasons, "samples": len(rows),
                "samples_total": total, "window": "samples timestamped inside the timed region only",
                "sample_period_ms": self.PERIOD_MS, "power_cap_frac": capped / len(rows),
                "power_w_instant_median": statistics.median(power) if power else None,
                "power_w_instant_max": max(power) if power else None}


# ----------------------------------------------------------------------------- the CUDA arm

def traffic_record(kind, workload, path):
    """DRAM bytes per launch of `kind` on `path` from a committed ncu capture, if it was
    taken on the kernel source as it is now (else None)."""
    rec = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(rec) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None
    src = os.path.join(ROOT, "lm_head_cross_gb300", "csrc", "flce_kernels.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for r in recs:
        if (r.get("kind") == kind and r.get("workload") == workload and r.get("path", "rowchunk") == path
                and r.get("kernel_sha") == sha):
            return float(r["bytes_per_launch"])
    return None


def device_problem(name, rank, dev):
    import numpy as np
    import torch
    import synth
    c = dict(synth.WORKLOADS[name])
    c["seed"] = rank_seed(c["seed"], rank)
    problem = synth.make_problem(**c)
    X = torch.from_numpy(problem.X.view(np.int16)).view(torch.bfloat16).to(dev)
    W = torch.from_numpy(problem.W.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.from_numpy(problem.labels).to(dev)
    return problem, X, W, y


def ws_bytes_of(flce, rowchunk, problem, reduction=None):
    f = flce.workspace_bytes_rowchunk if rowchunk else flce.workspace_bytes
    return f(problem.n, problem.h, problem.v, problem.ignore_index, reduction or problem.reduction)


def extra_memory(flce, torch, dev, X, W, y, problem, rowchunk):
    """Device memory one call allocates beyond its inputs and outputs (the torch allocator's
    peak delta), next to the workspace size the library asks for; fails on a device error."""
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    tmp = flce.fwd_bwd(X, W, y, problem.ignore_index, problem.reduction, rowchunk=rowchunk)
    torch.cuda.synchronize()
    out_bytes = sum(t.numel() * t.element_size() for t in tmp[:4])
    peak = torch.cuda.max_memory_allocated(dev) - base - out_bytes
    st = flce.read_device_status(tmp[4])
    del tmp
    if st != 0:
        raise RuntimeError(f"device status {flce.status_string(st)}")
    return int(peak)


def timed_steps(step, steps, warmup, flush, stream, torch, flce, clocks=None, dist=None):
    """W >= 3 untimed steps, then K steps each bracketed by CUDA events on the launching
    stream, a 512 MiB write between steps (outside the events) to evict L2; the dominant
    kernel kind is timed live by the library's own events around its launches."""
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in starts + ends:      # create the driver events now, not inside the timed loop
        e.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    flce.profile_enable(True, kinds=["dxdw"])   # the dominant kernel only: events elsewhere would serialise launches
    if clocks is not None:
        clocks.mark_start()
    t_wall0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if clocks is not None:
        clocks.mark_end()
    if dist is not None:
        dist.barrier()
    dom = flce.profile_read()["dxdw"]
    flce.profile_enable(False)
    return {"step_ms": [a.elapsed_time(b) for a, b in zip(starts, ends)], "dom": dom, "wall_s": t_wall}


def dominant_tflops(dom):
    n_l, ms_l, fl_l = dom
    return (fl_l / n_l) / ((ms_l / n_l) / 1e3) / 1e12 if n_l and ms_l else None


def measure_path(flce, torch, dev, problem, X, W, y, rowchunk, steps, warmup, flush, stream, naive=False):
    """One (workload, path) measured with the headline's timing discipline: credited and
    executed TFLOP/s, the dominant kernel's rate, extra device memory."""
    wsb = ws_bytes_of(flce, rowchunk, problem)
    peak = extra_memory(flce, torch, dev, X, W, y, problem, rowchunk)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    out = (torch.empty(1, dtype=torch.float32, device=dev), torch.empty(problem.n, dtype=torch.float32, device=dev),
           torch.empty_like(X), torch.empty_like(W))

    def step():
        flce.fwd_bwd(X, W, y, problem.ignore_index, problem.reduction, ws=ws, out=out, rowchunk=rowchunk)

    r = timed_steps(step, steps, warmup, flush, stream, torch, flce)
    st = flce.read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {flce.status_string(st)}")
    ms = sum(r["step_ms"]) / steps
    n, h, v = problem.n, problem.h, problem.v
    res = {"path": "rowchunk (6NHV executed)" if rowchunk else "bounded (8NHV executed)",
           "value": credited_flops(n, h, v) / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": ms, "steps": steps,
           "executed_tflops": (6.0 if rowchunk else 8.0) * n * h * v / (ms / 1e3) / 1e12,
           "dominant_kernel_tflops": dominant_tflops(r["dom"]), "extra_hbm_bytes": wsb,
           "peak_alloc_delta_bytes": peak}
    del ws, out
    if naive:
        res["torch_naive"] = torch_naive(X, W, y, problem, flush, stream, torch)
    return res


def e2e_measure(args, flce, torch, dev, dist, problem, X, W, y, out, stream, world, flops):
    """End to end through the public C-ABI call on host memory (flce_fwd_bwd_host, the
    bounded path): every step copies its inputs in and its results out; the copies run on
    their own streams and two device buffers alternate, so one step's copies overlap the
    neighbouring steps' kernels while the kernels stay in order on one stream."""
    n, h, v = problem.n, problem.h, problem.v
    Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True); Xh.copy_(X)
    Wh = torch.empty(W.shape, dtype=W.dtype, pin_memory=True); Wh.copy_(W)
    yh = torch.empty(y.shape, dtype=y.dtype, pin_memory=True); yh.copy_(y)
    hb = flce.host_buffer_bytes(n, h, v, problem.ignore_index, problem.reduction)
    comp, cin, cout = (torch.cuda.Stream(device=dev) for _ in range(3))
    slots = [(tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in out),
              torch.empty(hb, dtype=torch.uint8, device=dev), torch.cuda.Event()) for _ in range(2)]

    def e2e_run(steps):
        for i in range(steps):
            outs, buf, done = slots[i % 2]
            if i >= 2:
                cin.wait_event(done)  # the previous call on this buffer has copied its results out
            flce.fwd_bwd_host(Xh, Wh, yh, outs, buf, problem.ignore_index, problem.reduction, stream=comp,
                              in_stream=cin, out_stream=cout)
            done.record(cout)

    e2e_run(2)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    clocks.mark_start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st_ in (comp, cin, cout):
        st_.wait_event(e0)
    e2e_run(args.e2e_steps)
    for st_ in (comp, cin, cout):
        fin = torch.cuda.Event()
        fin.record(st_)
        stream.wait_event(fin)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop() or {}
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    for _, buf, _ in slots:
        st_code = flce.read_device_status(buf)
        if st_code != 0:
            raise RuntimeError(f"device status {flce.status_string(st_code)}")
    del slots, Xh, Wh, yh
    h2d = sum(t.numel() * t.element_size() for t in (X, W, y))
    d2h = sum(t.numel() * t.element_size() for t in out)

    e2e_value = job_tflops(world, flops, args.e2e_steps, e2e_ms)
    return {"value": e2e_value, "unit": UNIT,
            "tflops_per_ghz": e2e_value / world / (clk["sm_mhz"] / 1e3) if clk.get("sm_mhz") else None,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_mhz_min", "reasons", "samples", "power_cap_frac",
                                               "power_w_instant_median")},
            "note": "flce_fwd_bwd_host (bounded path) through the C-ABI: pinned host X, W, labels copied in "
                    "and loss, lse, dX, dW copied out every step, on their own streams; two device buffers "
                    "alternate so copies overlap the neighbouring steps' kernels"}


def run_flce(args, rank, world, local_rank):
    import torch
    import lm_head_cross_gb300 as flce

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    problem, X, W, y = device_problem(args.workload, rank, dev)
    n, h, v = problem.n, problem.h, problem.v
    rowchunk = args.path == "rowchunk"
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    reduction = args.reduction or problem.reduction
    ws_bytes = ws_bytes_of(flce, rowchunk, problem, reduction)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = (torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=dev),
           torch.empty(n, dtype=torch.float32, device=dev), torch.empty_like(X), torch.empty_like(W))

    if args.op == "fwd_bwd":
        seq = n if args.shift else 0

        def step():
            flce.fwd_bwd(X, W, y, problem.ignore_index, reduction, ws=ws, out=out, shift=args.shift, seq_len=seq,
                         rowchunk=rowchunk)
    elif args.op == "topk":
        tk_ws = torch.empty(flce.topk_workspace_bytes(n, h, v, args.k), dtype=torch.uint8, device=dev)

        def step():
            flce.topk(X, W, args.k, ws=tk_ws)
    else:
        g = torch.Generator(device="cpu").manual_seed(5)
        sidx = torch.stack([torch.randperm(v, generator=g)[:args.k] for _ in range(min(n, 64))])
        sidx = sidx.repeat((n + 63) // 64, 1)[:n].to(torch.int32).contiguous().to(dev)
        sq = torch.softmax(torch.randn(n, args.k, generator=g), dim=1).to(torch.float32).contiguous().to(dev)

        def step():
            flce.soft_fwd_bwd(X, W, sidx, sq, reduction, ws=ws, rowchunk=rowchunk)

    if args.op != "fwd_bwd" or args.reduction or args.shift:
        return run_variant(args, step, n, h, v, world, dev, dist, torch, flce, flush, stream)

    # extra device memory of one call beyond its inputs and outputs: the workspace, up to the
    # caching allocator's rounding (512-byte sizes; a reused cached block that is not split
    # keeps up to 1 MiB of slack per allocation, five allocations per call)
    peak_delta = extra_memory(flce, torch, dev, X, W, y, problem, rowchunk)
    if not ws_bytes <= peak_delta <= ws_bytes + (5 << 20) + 4096:
        raise RuntimeError(f"allocation beyond the workspace: peak delta {peak_delta} vs workspace {ws_bytes}")
    if args.workload == HEADLINE and not rowchunk and ws_bytes >= 4e9:
        raise RuntimeError(f"workspace of the 128K x 128K workload is {ws_bytes} bytes, not under 4 GB")

    clocks = ClockSampler(local_rank)
    clocks.start()
    r = timed_steps(step, args.steps, args.warmup, flush, stream, torch, flce, clocks=clocks, dist=dist)
    clk = clocks.stop() or {"reasons": ["no sampler"], "samples": 0}
    st = flce.read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {flce.status_string(st)}")
    prof, per_step = kernel_breakdown(flce, torch, step, flush, min(args.steps, 5))
    step_ms = r["step_ms"]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    flops = credited_flops(n, h, v)
    value = job_tflops(world, flops, args.steps, total_ms)

    e2e = None
    if args.e2e_steps > 0:
        e2e = e2e_measure(args, flce, torch, dev, dist, problem, X, W, y, out, stream, world, flops)

    naive = None
    if rank == 0 and world == 1 and not args.no_naive:
        naive = torch_naive(X, W, y, problem, flush, stream, torch)

    # the other path on the same inputs, then both paths on the other workloads
    others = None
    if world == 1 and not args.no_others:
        del ws
        torch.cuda.empty_cache()
        others = {"other_path": measure_path(flce, torch, dev, problem, X, W, y, not rowchunk, args.other_steps, 3,
                                             flush, stream)}
        del X, W, y, out
        torch.cuda.empty_cache()
        wl = {}
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            p_o, X_o, W_o, y_o = device_problem(name, rank, dev)
            wl[name] = {"bounded": measure_path(flce, torch, dev, p_o, X_o, W_o, y_o, False, args.other_steps, 3,
                                                flush, stream),
                        "rowchunk": measure_path(flce, torch, dev, p_o, X_o, W_o, y_o, True, args.other_steps, 3,
                                                 flush, stream, naive=not args.no_naive)}
            del X_o, W_o, y_o, p_o
            torch.cuda.empty_cache()
        others["workloads"] = wl

    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peaks, peak_src = load_peaks()
    kinds = {k: {"launches": n_, "ms": ms_, "tflop": fl_ / 1e12} for k, (n_, ms_, fl_) in prof.items()}
    dom = "dxdw"
    achieved = dominant_tflops(r["dom"])
    peak_sust = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # a timed region whose median SM clock stayed at the maximum is compared with the burst
    # peak, one that the power cap held lower (a long, heavy run) with the sustained peak
    capped = bool(clk.get("sm_mhz") and clk.get("sm_max_mhz") and clk["sm_mhz"] < 0.95 * clk["sm_max_mhz"])
    peak, peak_kind = (peak_sust, "bf16_tflops_sustained") if capped else (peak_burst, "bf16_tflops (burst)")
    path_name = "rowchunk" if rowchunk else "bounded"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": arm_config(args, world),
        "frac_of_peak": value / world / peak_burst, "frac_of_sustained_peak": value / world / peak_sust,
        "peak_src": f"{peak_src} bf16_tflops (burst) / bf16_tflops_sustained",
        "executed_tflops": world * per_step["flops"] * args.steps / (total_ms / 1e3) / 1e12,
        "path": ("row chunks, logits computed once (6NHV executed); workspace grows with V" if rowchunk else
                 "bounded: logits recomputed per vocabulary chunk in the backward (8NHV executed); "
                 "workspace independent of V"),
        "extra_hbm_bytes": ws_bytes, "peak_alloc_delta_bytes": int(peak_delta),
        "materialised_logits_bytes": {"bf16": flce.logits_footprint_bytes(n, v, 2),
                                      "fp32": flce.logits_footprint_bytes(n, v, 4)},
        "timed_region_s": sum(step_ms) / 1e3,
        "wall_ms_per_step_incl_flush": 1e3 * r["wall_s"] / args.steps,
        "step_ms_min_median_max": [min(step_ms), statistics.median(step_ms), max(step_ms)],
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "peak_note": f"{peak_src} {peak_kind} ({'power-capped' if capped else 'full clock'} during the "
                                  f"timed region); of burst {peak_burst}: {achieved / peak_burst:.3f}, of sustained "
                                  f"{peak_sust}: {achieved / peak_sust:.3f}",
                     "algorithmic_flops_per_launch": r["dom"][2] / r["dom"][0],
                     "launches_timed": r["dom"][0],
                     "traffic": traffic_record(dom, args.workload, path_name)},
        "kernels": kinds,
        "kernels_note": "separate untimed pass with every launch bracketed by events (which serialises the "
                        "launches); the roofline kernel is timed inside the timed region",
        "gpu_launches": per_step["launches"] * args.steps,
        "clocks": clk,
        "tflops_per_ghz": (value / world) / (clk["sm_mhz"] / 1e3) if clk.get("sm_mhz") else None,
        "e2e": e2e,
    }
    if naive is not None:
        line["torch_naive"] = naive
    if others is not None:
        line["other_path"] = others["other_path"]
        line["workloads"] = others["workloads"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(problem, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def kernel_breakdown(flce, torch, step, flush, steps):
    """Per-kind launch counts and device times from a separate pass in which
    every launch is bracketed by events; also the launches and flops per step."""
    flce.profile_enable(True)
    for i in range(steps):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    prof = flce.profile_read()
    flce.profile_enable(False)
    per_step = {"launches": sum(x[0] for x in prof.values()) // steps,
                "flops": sum(x[2] for x in prof.values()) / steps}
    return prof, per_step


def run_variant(args, step, n, h, v, world, dev, dist, torch, flce, flush, stream):
    """A non-default operation or option: same timing discipline, its own metric line."""
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in starts + ends:
        e.record(stream)
    torch.cuda.synchronize()
    dom = "forward" if args.op == "topk" else "dxdw"
    flce.profile_enable(True, kinds=[dom])
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    clocks.mark_start()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clk = clocks.stop() or {"reasons": ["no sampler"], "samples": 0}
    prof_dom = flce.profile_read()[dom]
    flce.profile_enable(False)
    prof, per_step = kernel_breakdown(flce, torch, step, flush, min(args.steps, 10))
    total_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)), dist, dev)
    credited = (2.0 if args.op == "topk" else 6.0) * n * h * v
    if dist is not None:
        dist.destroy_process_group()
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    peaks, peak_src = load_peaks()
    value = job_tflops(world, credited, args.steps, total_ms)
    names = {"fwd_bwd": "fused linear-CE fwd+bwd TFLOP/s (6NHV)", "topk": "per-row top-k logits TFLOP/s (2NHV)",
             "soft": "fused linear + sparse-target KL fwd+bwd TFLOP/s (6NHV)"}
    print(json.dumps({
        "metric": names[args.op], "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(args.workload, None, f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
                                       world), op=args.op, k=args.k, reduction=args.reduction, shift=args.shift),
        "frac_of_peak": value / world / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
        "peak_src": peak_src,
        "dominant_kernel": {"kind": dom, "launches": prof_dom[0], "ms": prof_dom[1],
                            "tflops": prof_dom[2] / (prof_dom[1] / 1e3) / 1e12 if prof_dom[1] else None},
        "kernels": {k: {"launches": a, "ms": b, "tflop": c / 1e12} for k, (a, b, c) in prof.items()},
        "gpu_launches": per_step["launches"] * args.steps,
        "clocks": clk,
    }), flush=True)
    return 0


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_flce(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
