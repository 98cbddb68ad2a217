#!/usr/bin/env python3
"""Benchmark of triangular attention forward + backward on GB300.

One step = tri_attn_fwd + tri_attn_bwd (preprocess, key-tile-parallel main
kernel, dQ and dbias reductions) over one batch of seeded synthetic BF16
inputs of the headline crop (B=1, N=N_o=768, H=4, D=32, last 8% of keys
masked).  FLOPs follow the convention fwd = 4U, bwd = 10U (five GEMMs with
the S recompute), step = 14U, U = B*N_o*H*N*N*D.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the FP64 CPU
oracle instead (the only reference this path has; it is a deliberately slow
program, so the ratio is context, not a headline).

Multi-GPU (torchrun): every rank runs its own independent problem of the
same shape (the method's slices are independent; no data-path collective),
so scaling is weak and ``value`` is the total over all ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tri-attn fwd+bwd TFLOP/s (N=768 H=4 D=32)"


def metric_for(w) -> str:
    """The headline metric's name on its own workload; other workloads name
    their shape in the same form."""
    if (w.B, w.N, w.H, w.D) == (1, 768, 4, 32):
        return METRIC
    return f"tri-attn fwd+bwd TFLOP/s (B={w.B} N={w.N} H={w.H} D={w.D})"
UNIT = "TFLOP/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="crop768")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--calls", type=int, default=100,
                    help="individually timed fwd / bwd calls (after 10 warm-ups) for the median and mean")
    ap.add_argument("--ablation", choices=["atomic"], default=None,
                    help="instead of the bench line: time the ordered backward against its non-deterministic "
                         "variants (FP32 atomics for dQ, dbias, both; TMA bulk reduction for dQ) on the same inputs and print one "
                         "JSON line")
    ap.add_argument("--module", type=int, default=0, metavar="C",
                    help="instead of the bench line: time the whole module (LayerNorm, projections with C pair "
                         "features, the core, output projection; forward + backward) and print one JSON line")
    ap.add_argument("--trimul", type=int, default=0, metavar="C",
                    help="instead of the bench line: time the triangle multiplicative update (C pair features = "
                         "C hidden channels, forward + backward, both directions) and print one JSON line each")
    return ap.parse_args()


def flops(w):
    U = w.B * w.No * w.H * w.N * w.N * w.D
    return 4 * U, 10 * U, 14 * U


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"bf16_burst": d.get("bf16_tflops", 1900.0), "bf16_sustained": d.get("bf16_tflops_sustained", 1700.0),
                "hbm_gbs": d.get("hbm_gbs", 6800.0), "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"triattn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        try:
            self.f.close()
        except Exception:
            pass

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_ranks(local_ms: float, flop_per_step: int, steps: int, world: int, device=None) -> tuple:
    """Max of the per-rank elapsed times over all ranks (the slowest rank
    defines the job's time) and the whole-job throughput in TFLOP/s: every
    rank processed `steps` steps of its own problem."""
    import torch
    import torch.distributed as dist
    ms = float(local_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, flop_per_step * steps * world / (ms * 1e-3) / 1e12


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "tri_attn_fwd": ["protein_folding_triangle_gb300/csrc/fwd.cu", "protein_folding_triangle_gb300/csrc/ptx.cuh"],
    "fwd_prep": ["protein_folding_triangle_gb300/csrc/fwd.cu"],
    "bwd_main": ["protein_folding_triangle_gb300/csrc/bwd.cu", "protein_folding_triangle_gb300/csrc/ptx.cuh"],
    "bwd_preprocess": ["protein_folding_triangle_gb300/csrc/bwd.cu"],
    "bwd_transpose_bias": ["protein_folding_triangle_gb300/csrc/bwd.cu"],
    "bwd_reduce_dq": ["protein_folding_triangle_gb300/csrc/bwd.cu"],
    "bwd_reduce_dbias": ["protein_folding_triangle_gb300/csrc/bwd.cu"],
}


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


def kernel_work(w, name):
    """Algorithmic work per launch: (amount, unit, bound)."""
    U = w.B * w.No * w.H * w.N * w.N * w.D
    rows = w.B * w.No * w.H * w.N
    jk = (w.N + 127) // 128
    groups = w.No // (8 if w.D == 16 else 4)  # outer slices per backward CTA
    if name == "tri_attn_fwd":
        return 4 * U, "flop", "tensor"
    if name == "fwd_prep":  # key mask in, 144-byte records out (+ the padded bias when N % 8 != 0)
        jk64 = (w.N + 63) // 64
        pad = 2 * w.B * w.H * w.N * ((w.N + 7) // 8 * 8) * 2 if w.N % 8 else 0
        return w.B * w.No * w.N * 2 + (w.B * w.No + 4) * jk64 * 144 + pad, "byte", "hbm"
    if name == "bwd_main":
        return 10 * U, "flop", "tensor"
    if name == "bwd_preprocess":
        jq = (w.N + 127) // 128
        return 3 * rows * w.D * 2 + rows * 4 + w.B * w.No * w.H * jq * 128 * 16, "byte", "hbm"
    if name == "bwd_transpose_bias":
        return 2 * w.B * w.H * w.N * w.N * 2, "byte", "hbm"
    if name == "bwd_reduce_dq":
        return jk * rows * w.D * 4 + rows * w.D * 2, "byte", "hbm"
    if name == "bwd_reduce_dbias":
        return groups * w.B * w.H * w.N * w.N * 4 + w.B * w.H * w.N * w.N * 2, "byte", "hbm"
    raise KeyError(name)


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(w, x, seconds: float, gpu_out=None):
    """Time the FP64 oracle (fwd + bwd) on a bounded sample of the workload:
    the first n outer slices of example 0, all heads.  Returns the
    cpu_baseline dict and, if GPU outputs are given, the relative RMSE of the
    GPU's O, dQ, dK and dV on the sampled slices."""
    import numpy as np
    from oracle import oracle as O

    O.build()

    def run(n):
        sub = {k: (None if v is None else v[:1, :n].contiguous()) for k, v in x.items() if k != "bias"}
        bias = x["bias"][:1]
        t0 = time.perf_counter()
        o, lse = O.fwd(sub["q"], sub["k"], sub["v"], bias, sub["mask"])
        dq, dk, dv, _ = O.bwd(sub["q"], sub["k"], sub["v"], bias, sub["mask"], sub["do"])
        return time.perf_counter() - t0, {"o": o, "dq": dq, "dk": dk, "dv": dv}

    # calibrate on enough slices to keep every core busy (the oracle runs
    # (slice, head) items in parallel), so the estimate scales to the sample
    n_cal = int(min(w.No, 16))
    t_cal, _ = run(n_cal)
    per_slice = t_cal / n_cal
    n = int(max(2, min(w.No, seconds / max(per_slice, 1e-6))))
    dt, ref = run(n)
    U = 1 * n * w.H * w.N * w.N * w.D
    value = 14 * U / dt / 1e12
    res = {"value": value, "unit": UNIT, "cores": O.max_threads(), "cpu": cpu_model(), "kind": "oracle",
           "sample": f"FP64 oracle fwd+bwd on outer slices 0..{n - 1} of example 0, all {w.H} heads "
                     f"({n}/{w.No * w.B} slices, {dt:.1f} s; 14*U FLOP convention)",
           "seconds": dt}
    rm = None
    if gpu_out is not None:
        def rel(a, r):
            a = a[:1, :n].float().cpu().double().numpy()
            return float(np.sqrt(np.mean((a - r) ** 2)) / np.sqrt(np.mean(r ** 2)))
        rm = {k: rel(gpu_out[k], ref[k]) for k in ("o", "dq", "dk", "dv")}
    return res, rm


def cpu_model() -> str:
    """The host CPU's model as /proc/cpuinfo names it (x86: "model name"; Arm:
    implementer and part numbers), else the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} (CPU implementer {fields.get('CPU implementer', '?')}, part {fields['CPU part']})"
    return platform.machine()


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import torch  # noqa: F401
    from protein_folding_triangle_gb300 import synthetic as S
    w = S.WORKLOADS[args.workload]
    x = S.make_inputs(w, seed=args.seed)
    per_step = []
    info = None
    budget = max(2.0, args.cpu_seconds / max(args.steps + args.warmup, 1))
    for i in range(args.warmup + args.steps):
        res, _ = oracle_sample(w, x, budget)
        if i >= args.warmup:
            per_step.append(res)
            info = res
    val = statistics.median(r["value"] for r in per_step)
    line = {"metric": metric_for(w), "value": val, "unit": UNIT, "impl": "reference", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.describe(), "B": w.B, "N": w.N, "H": w.H, "D": w.D},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": info["cores"], "cpu": info["cpu"],
                             "kind": "oracle", "sample": info["sample"]},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args):
    import torch
    import torch.distributed as dist
    from protein_folding_triangle_gb300 import build as B
    from protein_folding_triangle_gb300 import synthetic as S
    from protein_folding_triangle_gb300 import triattn as T

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local if ws > 1 else 0)
    B.build()
    T.load()
    w = S.WORKLOADS[args.workload]
    x = S.make_inputs(w, seed=args.seed + rank)
    xd = {k: (None if v is None else v.to(dev)) for k, v in x.items()}
    stream = torch.cuda.current_stream(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base_mem = torch.cuda.memory_allocated(dev)
    o = torch.empty_like(xd["q"])
    lse = torch.empty(xd["q"].shape[:-1], dtype=torch.float32, device=dev)
    resid = torch.empty_like(xd["q"])
    dq, dk, dv = torch.empty_like(xd["q"]), torch.empty_like(xd["q"]), torch.empty_like(xd["q"])
    dbias = torch.empty_like(xd["bias"])
    wsb = torch.empty(T.bwd_workspace_bytes(xd["q"]), dtype=torch.uint8, device=dev)
    wsf = torch.empty(max(T.fwd_workspace_bytes(xd["q"]), 256), dtype=torch.uint8, device=dev)

    def step(inp):
        T.tri_attn_fwd(inp["q"], inp["k"], inp["v"], inp["bias"], inp["mask"], out=(o, lse, resid), workspace=wsf)
        T.tri_attn_bwd(inp["q"], inp["k"], inp["v"], inp["bias"], inp["mask"], o, resid, lse, inp["do"],
                       workspace=wsb, out=(dq, dk, dv, dbias))

    def barrier():
        if ws > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step(xd)
    torch.cuda.synchronize(dev)
    if T.device_status() != T.OK:
        raise SystemExit("device status not OK after warm-up")

    # ---------------- device-timed region (inputs resident in HBM)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        T.trace_enable(True)
        e0.record(stream)
        for _ in range(args.steps):
            step(xd)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        T.trace_enable(False)
        barrier()
    trace = T.trace_read()
    peak_mem = torch.cuda.max_memory_allocated(dev) - base_mem
    f_fwd, f_bwd, f_step = flops(w)
    ms, value = combine_ranks(e0.elapsed_time(e1), f_step, args.steps, ws, dev)

    # ---------------- end-to-end: pinned host buffers, copies inside the timed region
    # Every step copies its own inputs host -> device and reads its four
    # gradients back device -> host.  As in a training loop, the copies of
    # neighbouring steps overlap the compute: host->device copies on one
    # stream, compute on another, device->host on a third; inputs and
    # gradients are double-buffered and every reuse of a buffer waits on the
    # event of its last user.
    e2e = None
    if not args.no_e2e:
        hx = {k: (None if v is None else v.pin_memory()) for k, v in x.items()}
        names = ("dq", "dk", "dv", "dbias")
        hgrads = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv, dbias)]
        h2d = sum(v.numel() * v.element_size() for v in hx.values() if v is not None)
        d2h = sum(t.numel() * t.element_size() for t in hgrads)
        dx = [{k: (None if v is None else torch.empty_like(xd[k])) for k, v in hx.items()} for _ in range(2)]
        dgrads = [[torch.empty_like(t) for t in (dq, dk, dv, dbias)] for _ in range(2)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b copied
        ev_cmp = [torch.cuda.Event() for _ in range(2)]    # step on buffer b done
        ev_out = [torch.cuda.Event() for _ in range(2)]    # gradients of buffer b copied out
        used = [False, False]

        def e2e_steps(n):
            for k in range(n):
                bi = k & 1
                with torch.cuda.stream(s_in):
                    if used[bi]:
                        s_in.wait_event(ev_cmp[bi])        # step k-2 no longer reads these inputs
                    for key, v in hx.items():
                        if v is not None:
                            dx[bi][key].copy_(v, non_blocking=True)
                    ev_in[bi].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in[bi])
                    if used[bi]:
                        s_cmp.wait_event(ev_out[bi])       # gradients of step k-2 copied out
                    inp = dx[bi]
                    T.tri_attn_fwd(inp["q"], inp["k"], inp["v"], inp["bias"], inp["mask"], out=(o, lse, resid),
                                   workspace=wsf)
                    T.tri_attn_bwd(inp["q"], inp["k"], inp["v"], inp["bias"], inp["mask"], o, resid, lse, inp["do"],
                                   workspace=wsb, out=tuple(dgrads[bi]))
                    ev_cmp[bi].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[bi])
                    for hg, g in zip(hgrads, dgrads[bi]):
                        hg.copy_(g, non_blocking=True)
                    ev_out[bi].record(s_out)
                used[bi] = True

        e2e_steps(2)
        torch.cuda.synchronize(dev)
        barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        s_cmp.wait_stream(s_in)
        s_out.wait_stream(s_in)
        e2e_steps(args.steps)
        s_in.wait_stream(s_cmp)
        s_in.wait_stream(s_out)
        a1.record(s_in)
        torch.cuda.synchronize(dev)
        ems, evalue = combine_ranks(a0.elapsed_time(a1), f_step, args.steps, ws, dev)
        e2e = {"value": round(evalue, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(ems / args.steps, 4),
               "copies": "overlapped with neighbouring steps (3 streams, double-buffered)"}
    # ---------------- per-call times: each call bracketed by its own events
    # (after 10 warm-up calls), median and mean over --calls calls
    per_call = None
    if args.calls > 0:
        for _ in range(10):
            step(xd)
        torch.cuda.synchronize(dev)
        tf, tb = [], []
        for _ in range(args.calls):
            c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            c0.record(stream)
            T.tri_attn_fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], out=(o, lse, resid), workspace=wsf)
            c1.record(stream)
            T.tri_attn_bwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], o, resid, lse, xd["do"],
                           workspace=wsb, out=(dq, dk, dv, dbias))
            c2.record(stream)
            c2.synchronize()
            tf.append(c0.elapsed_time(c1))
            tb.append(c1.elapsed_time(c2))
        ts = [a + b for a, b in zip(tf, tb)]
        per_call = {"calls": args.calls, "warmup_calls": 10}
        for name, v, fl in (("fwd", tf, f_fwd), ("bwd", tb, f_bwd), ("fwd_bwd", ts, f_step)):
            med, mean = statistics.median(v), statistics.mean(v)
            per_call[name] = {"median_ms": round(med, 4), "mean_ms": round(mean, 4),
                              "tflops_at_median": round(fl / (med * 1e-3) / 1e12, 2)}
    if T.device_status() != T.OK:
        raise SystemExit("device status not OK after timing")

    if rank != 0:
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    pk = peaks()
    # per-kernel summary from the live trace
    kernels = {}
    total_k = sum(e["total_ms"] for e in trace.values())
    for name, e in trace.items():
        amount, unit, bound = kernel_work(w, name)
        mean_ms = e["mean_ms"]
        rate = amount / (mean_ms * 1e-3)
        kernels[name] = {"launches": e["launches"], "mean_ms": round(mean_ms, 4),
                         "share": round(e["total_ms"] / total_k, 4),
                         ("TFLOP/s" if unit == "flop" else "GB/s"): round(rate / (1e12 if unit == "flop" else 1e9), 2)}
    dom = max(trace, key=lambda n: trace[n]["total_ms"])
    amount, unit, bound = kernel_work(w, dom)
    dom_ms = trace[dom]["mean_ms"]
    # The timed region lasts well under a second (no sustained power-cap
    # regime), so a contraction is measured against the burst BF16 peak; a
    # region of seconds would take the sustained one.
    long_region = ms >= 1000.0
    if unit == "flop":
        achieved = amount / (dom_ms * 1e-3) / 1e12
        peak = pk["bf16_sustained"] if long_region else pk["bf16_burst"]
        runit = "TFLOP/s"
    else:
        achieved = amount / (dom_ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        runit = "GB/s"
    traffic = ncu_traffic(dom)
    fwd_ms = sum(trace[n]["mean_ms"] for n in ("fwd_prep", "tri_attn_fwd") if n in trace) or None
    bwd_ms = sum(trace[n]["mean_ms"] for n in ("bwd_preprocess", "bwd_transpose_bias", "bwd_main", "bwd_reduce_dq",
                                                "bwd_reduce_dbias")
                 if n in trace)
    clocks = clk.summary()
    # Secondary ceiling of the two main kernels: the exponentials of the
    # softmax (one exp2 per score in each) on the MUFU pipe, 32 per clock per
    # SM (measured on GB300), at the SM clock sampled during the timed region.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    mufu_peak = 32.0 * sms * mhz * 1e6
    scores = w.B * w.No * w.H * w.N * w.N
    secondary = {"bound": "mufu", "unit": "exp2/s", "peak": mufu_peak,
                 "peak_source": f"32 exp2 per clock per SM x {sms} SMs x {mhz} MHz"}
    for name in ("tri_attn_fwd", "bwd_main"):
        if name in trace:
            rate = scores / (trace[name]["mean_ms"] * 1e-3)
            secondary[name] = {"achieved": rate, "frac": round(rate / mufu_peak, 4)}
    line = {
        "metric": metric_for(w), "value": round(value, 3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.describe(), "B": w.B, "N": w.N, "N_o": w.No, "H": w.H, "D": w.D,
                   "seed": args.seed, "parallelism": f"replicas{ws}" if ws > 1 else "single",
                   "l2": "inputs larger than L2 (Q,K,V,dO,O,E 6x144 MiB + FP32 partials per step), no flush",
                   "flop_convention": "fwd 4U, bwd 10U, step 14U, U=B*N_o*H*N*N*D (dense keys)"},
        "fwd_tflops": round(f_fwd / (fwd_ms * 1e-3) / 1e12, 2) if fwd_ms else None,
        "bwd_tflops": round(f_bwd / (bwd_ms * 1e-3) / 1e12, 2) if bwd_ms else None,
        "frac_bf16_peak": {"sustained": round(value / ws / pk["bf16_sustained"], 4),
                           "burst": round(value / ws / pk["bf16_burst"], 4), "peaks": pk["source"]},
        "roofline": {"kernel": dom, "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{pk['source']} ("
                                    f"{('bf16 sustained' if long_region else 'bf16 burst') if unit == 'flop' else 'hbm copy'}"
                                    f"; timed region {ms:.0f} ms)"},
        "secondary": secondary,
        "kernels": kernels,
        "gpu_launches": sum(e["launches"] for e in trace.values()),
        "per_call": per_call,
        "peak_mem_bytes": int(peak_mem),
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        cb, rm = oracle_sample(w, x, args.cpu_seconds, gpu_out={"o": o, "dq": dq, "dk": dk, "dv": dv})
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "cpu", "kind", "sample")}
        line["rel_rmse_vs_fp64_on_sample"] = rm
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- ablation
def run_atomic_ablation(args):
    """Backward only: the ordered single-writer partials + fixed-order reductions
    against FP32 atomics for dQ, for dbias, and for both, and TMA bulk
    reductions for dQ (the pages' Table 12
    trade-off).  Same inputs, same launch stream, CUDA events, median of
    ``--steps`` timed calls after ``--warmup``; every call re-zeroes its
    accumulators, as a training step would."""
    import statistics
    import torch
    from protein_folding_triangle_gb300 import build as B
    from protein_folding_triangle_gb300 import synthetic as S
    from protein_folding_triangle_gb300 import triattn as T

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    B.build()
    T.load()
    dev = torch.device("cuda", 0)
    w = S.WORKLOADS[args.workload]
    xd = {k: (None if v is None else v.to(dev)) for k, v in S.make_inputs(w, seed=args.seed).items()}
    o, lse, resid = T.tri_attn_fwd(xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"])
    outs = (torch.empty_like(xd["q"]), torch.empty_like(xd["q"]), torch.empty_like(xd["q"]), torch.empty_like(xd["bias"]))
    arms = {"ordered": None, "atomic_dq": T.ATOMIC_DQ, "atomic_dbias": T.ATOMIC_DBIAS,
            "atomic_dbias_dq": T.ATOMIC_DBIAS_DQ, "bulk_dq": T.BULK_DQ, "bulk_dq_atomic_dbias": T.BULK_DQ_ATOMIC_DBIAS}
    wsb = {}
    for name, m in arms.items():
        need = T.bwd_workspace_bytes(xd["q"]) if m is None else T.bwd_atomic_workspace_bytes(xd["q"], m)
        wsb[name] = torch.empty(need, dtype=torch.uint8, device=dev)

    def call(name):
        m = arms[name]
        args_ = (xd["q"], xd["k"], xd["v"], xd["bias"], xd["mask"], o, resid, lse, xd["do"])
        if m is None:
            T.tri_attn_bwd(*args_, workspace=wsb[name], out=outs)
        else:
            T.tri_attn_bwd_atomic_ablation(*args_, m, workspace=wsb[name], out=outs)

    times = {n: [] for n in arms}
    for _ in range(max(3, args.warmup)):
        for n in arms:
            call(n)
    torch.cuda.synchronize(dev)
    for _ in range(args.steps):
        for n in arms:  # interleaved, so that clock drift hits every arm alike
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call(n)
            e1.record()
            e1.synchronize()
            times[n].append(e0.elapsed_time(e1))
    if T.device_status() != T.OK:
        raise SystemExit("device status not OK after the ablation")
    med = {n: statistics.median(v) for n, v in times.items()}
    line = {"ablation": "ordered FP32 partials vs FP32 atomics and TMA bulk reductions (backward only)",
            "config": {"workload": w.describe(), "B": w.B, "N": w.N, "H": w.H, "D": w.D},
            "steps": args.steps, "warmup": max(3, args.warmup),
            "bwd_ms_median": {n: round(v, 4) for n, v in med.items()},
            "saving_vs_ordered": {n: round(1.0 - med[n] / med["ordered"], 4) for n in arms if n != "ordered"},
            "deterministic": {n: n == "ordered" for n in arms},
            "pages_table12_context": "atomic dbias saves 2.8-8.0% of the backward on the pages' GPUs"}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- module
def run_module(args):
    """Forward + backward of the module around the core on the workload's
    shape with ``--module`` pair features: CUDA events around each step on the
    launching stream, then one traced step for the per-kernel split.  The
    module's own kernels are HBM-bound; their algorithmic bytes per step are
    counted below from the tensors each one must read and write once."""
    import statistics
    import torch
    from protein_folding_triangle_gb300 import build as B
    from protein_folding_triangle_gb300 import synthetic as S
    from protein_folding_triangle_gb300 import triattn as T

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    B.build()
    T.load()
    dev = torch.device("cuda", 0)
    w = S.WORKLOADS[args.workload]
    C, H, D, N, Bn = args.module, w.H, w.D, w.N, w.B
    x = S.make_module_inputs(Bn, N, C, H, D, seed=args.seed, mask_frac=w.mask_frac if w.mask != "none" else 0.0)
    xd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    nctx, nws = T.module_sizes(Bn, N, C, H, D)
    ctx = torch.empty(nctx, dtype=torch.uint8, device=dev)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    out = torch.empty_like(xd["z"])
    F = 3 * H * D + H
    f32 = dict(dtype=torch.float32, device=dev)
    grads = (torch.empty_like(xd["z"]), torch.empty(C, **f32), torch.empty(C, **f32), torch.empty((C, F), **f32),
             torch.empty((H * D, C), **f32))

    def step():
        T.tri_attn_module_fwd(xd["z"], xd["mask"], xd["ln_w"], xd["ln_b"], xd["w_in"], xd["w_o"], H, D, ctx=ctx,
                              workspace=ws, out=out)
        T.tri_attn_module_bwd(xd["z"], xd["mask"], xd["ln_w"], xd["w_in"], xd["w_o"], ctx, xd["d_out"], H, D,
                              workspace=ws, out=grads)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    times = []
    with ClockSampler(0) as clk:
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            step()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
    T.trace_enable(True)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    tr = T.trace_read()
    T.trace_enable(False)
    if T.device_status() != T.OK:
        raise SystemExit("device status not OK after the module bench")
    M, HD = Bn * N * N, H * D
    act = Bn * N * H * N * D * 2
    fl_core = flops(w)[2]
    gemm_flop = 3 * (2 * M * C * F + 2 * M * HD * C)  # forward, then dX and dW of each projection
    by = {"module_ln_fwd": M * C * 4 + M * 8,             # z in, x out, mean and rstd
          "module_ln_bwd": M * C * 6 + M * 8,             # z, dx (BF16) in, dz out, mean and rstd
          "module_layout": 2 * (7 * act + 2 * Bn * H * N * N * 2)}  # q k v o / do dq dk dv, bias and dbias planes
    pk = peaks()
    per = {}
    for name, e in tr.items():
        ms = e["total_ms"] / 3.0
        d = {"ms_per_step": round(ms, 4), "launches_per_step": e["launches"] // 3}
        if name in by:
            d["GB_per_s"] = round(by[name] / ms / 1e6, 1)
            d["hbm_frac_of_measured"] = round(by[name] / ms / 1e6 / pk["hbm_gbs"], 3)
        if name == "module_gemm":
            d["TFLOP_per_s"] = round(gemm_flop / ms / 1e9, 1)
        per[name] = d
    med = statistics.median(times)
    line = {"module": "LayerNorm -> projections -> triangle attention core -> output projection, fwd + bwd",
            "config": {"workload": w.describe(), "B": Bn, "N": N, "C": C, "H": H, "D": D,
                       "mask_frac": w.mask_frac if w.mask != "none" else 0.0},
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step_median": round(med, 4),
            "ms_per_step_min": round(min(times), 4),
            "core_share": round(sum(v["ms_per_step"] for k, v in per.items() if not k.startswith("module_")) / med, 3),
            "flop_per_step": {"core": fl_core, "projections": gemm_flop},
            "kernels": per, "clocks": clk.summary(), "peaks_source": pk["source"]}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- trimul
def run_trimul(args):
    """Forward + backward of the triangle multiplicative update on the
    workload's B and N with C_z = C_h = ``--trimul`` (the pages' Table 10
    shapes), each direction: CUDA events around each step on the launching
    stream, then three traced steps for the per-kernel split.  Algorithmic
    bytes of the HBM-bound kernels and FLOPs of the GEMMs per step are
    counted below."""
    import statistics
    import torch
    from protein_folding_triangle_gb300 import build as B
    from protein_folding_triangle_gb300 import synthetic as S
    from protein_folding_triangle_gb300 import triattn as T

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    B.build()
    T.load()
    dev = torch.device("cuda", 0)
    w = S.WORKLOADS[args.workload]
    Bn, N, C = w.B, w.N, args.trimul
    Cz = Ch = C
    x = S.make_trimul_inputs(Bn, N, Cz, Ch, seed=args.seed, pad_frac=0.0)
    xd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    F = 4 * Ch + Cz
    M = Bn * N * N
    f32 = dict(dtype=torch.float32, device=dev)
    pk = peaks()
    for direction in ("outgoing", "incoming"):
        nctx, nws = T.trimul_sizes(Bn, N, Cz, Ch, direction)
        ctx = torch.empty(nctx, dtype=torch.uint8, device=dev)
        ws = torch.empty(nws, dtype=torch.uint8, device=dev)
        out = torch.empty_like(xd["z"])
        grads = (torch.empty_like(xd["z"]), torch.empty(Cz, **f32), torch.empty(Cz, **f32), torch.empty((Cz, F), **f32),
                 torch.empty(Ch, **f32), torch.empty(Ch, **f32), torch.empty((Ch, Cz), **f32))

        def step():
            T.triattn_trimul_fwd(xd["z"], xd["mask"], xd["ln_in_w"], xd["ln_in_b"], xd["w_p"], xd["ln_out_w"],
                                 xd["ln_out_b"], xd["w_o"], direction, ctx=ctx, workspace=ws, out=out)
            T.triattn_trimul_bwd(xd["z"], xd["mask"], xd["ln_in_w"], xd["w_p"], xd["ln_out_w"], xd["w_o"], ctx,
                                 xd["d_out"], direction, workspace=ws, out=grads)

        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize(dev)
        times = []
        with ClockSampler(0) as clk:
            for _ in range(args.steps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                step()
                e1.record()
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
        T.trace_enable(True)
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        tr = T.trace_read()
        T.trace_enable(False)
        # input LayerNorm: fwd reads z, writes x and the statistics; bwd reads z, dx (BF16) and the statistics
        by = {"trimul_ln_in": M * Cz * 4 + 8 * M + M * Cz * 6 + 8 * M,
              # projection + gating: fwd reads x, writes a, b, g; bwd reads x, dA, dB, writes dp's 4 C_h columns
              "trimul_proj_gate": (M * Cz * 2 + 2 * M * Ch * 2 + M * Cz * 2) + (M * Cz * 2 + 2 * M * Ch * 2 + M * 4 * Ch * 2),
              # output LayerNorm: fwd reads X, writes y and the statistics; bwd reads X, dy (BF16), writes dX
              "trimul_ln_out": (2 * M * Ch * 2 + 8 * M) + (M * Ch * 2 + M * Ch * 2 + 8 * M + M * Ch * 2),
              "trimul_out_gate": 3 * M * Cz * 2 + 5 * M * Cz * 2}
        fl = {"trimul_proj_gemm": 3 * 2 * M * Ch * Cz + 2 * 2 * M * Cz * F,
              "trimul_contract_gemm": 3 * 2 * Bn * Ch * N ** 3}
        per = {}
        for name, e in tr.items():
            ms = e["total_ms"] / 3.0
            d = {"ms_per_step": round(ms, 4), "launches_per_step": e["launches"] // 3}
            if name in by:
                d["GB_per_s"] = round(by[name] / ms / 1e6, 1)
                d["hbm_frac_of_measured"] = round(by[name] / ms / 1e6 / pk["hbm_gbs"], 3)
            if name in fl:
                d["TFLOP_per_s"] = round(fl[name] / ms / 1e9, 1)
                d["tensor_frac_of_measured_sustained"] = round(fl[name] / ms / 1e9 / pk["bf16_sustained"], 3)
            per[name] = d
        med = statistics.median(times)
        line = {"trimul": direction, "what": "triangle multiplicative update, forward + backward",
                "config": {"B": Bn, "N": N, "C_z": Cz, "C_h": Ch, "mask": "none"},
                "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step_median": round(med, 4),
                "ms_per_step_min": round(min(times), 4), "flop_per_step": fl, "kernels": per,
                "clocks": clk.summary(), "peaks_source": pk["source"],
                "pages_table10_context_h100_ms": {"384/128": 1.32, "640/128": 3.33, "768/128": 4.78}}
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.trimul:
        run_trimul(args)
        return
    if args.module:
        run_module(args)
        return
    if args.ablation == "atomic":
        run_atomic_ablation(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
