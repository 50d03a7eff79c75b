#!/usr/bin/env python
"""Throughput of the FlashAttention-2 hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
the forward (fa_fwd: O and LSE) and the recompute backward (fa_bwd's three
launches: D/LSE preprocess, dK/dV pass, dQ pass), on the workload
bf16, causal, B=4, H=32, N=8192, d=80 (the only workload that takes the
backward too).  Throughput is credited TFLOP/s: forward 4*B*H*N^2*d/2 and
backward 10*B*H*N^2*d/2 per step (causal halves both), i.e. five GEMMs for
the backward even though the two-pass backward executes seven.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  With N > 1 (under torchrun) every rank runs
its own copy of the workload (independent heads need no exchange: weak
scaling, no collective on the data path) and the timing is the max over
ranks.  ``--impl reference`` times the float64 CPU oracle instead, on a
bounded sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 and fraction of dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the fwd+bwd bench workload)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size (small profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the forward-only timing of the other configurations (the 'configs' key)")
    ap.add_argument("--config-steps", type=int, default=50, help="timed forwards per configuration in 'configs'")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time only the forward of --workload (the forward-only configurations), one JSON line")
    ap.add_argument("--split", default="1", help="with --fwd-only: key-range splits (an integer, or 'auto')")
    ap.add_argument("--fp8v", action="store_true",
                    help="with --fwd-only: V in float8 e5m2, transposed, P cast to e5m2 (fa_fwd_fp8v)")
    ap.add_argument("--fp8v-lazy", action="store_true",
                    help="with --fp8v: the lazy running-max rule (FA_FP8V_LAZY_MAX) instead of the page's steps")
    ap.add_argument("--bwd-only", action="store_true",
                    help="time only the backward of --workload on --bwd-path, one JSON line")
    ap.add_argument("--bwd-path", choices=["auto", "two_pass", "fused"], default="auto")
    ap.add_argument("--softmax", default=None, metavar="WORKLOAD",
                    help="time the row-softmax kernel on a named softmax workload instead, one JSON line")
    ap.add_argument("--source-hash", default=None, metavar="KERNEL",
                    help="print the source hash that a traffic line for KERNEL must carry, and exit")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (weak scaling: one independent replica per rank)
# ---------------------------------------------------------------------------

def dist_init(backend: str):
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    rank = dist.get_rank() if world > 1 else 0
    return rank, world


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity with one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        dev = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        if dev.isdigit():
            cmd[1:1] = ["-i", dev]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if rows:
            first = rows[0][0]
            rows = [r for r in rows if r[0] == first]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


#: Dense bf16 tensor-core peak of one GB300 on paper (context next to the
#: measured figure).
NOMINAL_BF16_TFLOPS = 2250.0


def tensor_peak(peaks, peak_src, clk):
    """The bf16 tensor peak that kernels timed in this run are held against.

    The measured burst figure (a cuBLAS GEMM timed alone at full clock): every
    timed region of this bench lasts well under a second, and the clocks
    sampled during it show whether the SMs stayed at full clock.  If the
    median sampled SM clock fell below 95 % of the maximum, the burst figure
    is scaled by that ratio (tensor throughput follows the SM clock).  The
    sustained figure was measured at a clock far below the maximum under a
    seconds-long GEMM loop, which these kernels never see."""
    burst = peaks["bf16_tflops"]
    mhz = clk.get("sm_mhz") if clk else None
    mx = clk.get("sm_max_mhz") if clk else None
    if mhz and mx and mhz < 0.95 * mx:
        return round(burst * mhz / mx, 1), (f"{peak_src} bf16 burst x median sampled SM clock "
                                            f"({mhz:.0f} of {mx:.0f} MHz)")
    return burst, f"{peak_src} bf16 burst (timed region well under a second, SMs at full clock)"


#: Sources each kernel is compiled from (a change to any of them makes an
#: earlier DRAM-traffic capture of that kernel stale).
KERNEL_SOURCES = {
    "fwd": ("fa_fwd.cu", "ptx.cuh", "fa_internal.h"),
    "bwd_pre": ("fa_bwd.cu", "ptx.cuh", "fa_internal.h"),
    "bwd_dkdv": ("fa_bwd.cu", "ptx.cuh", "fa_internal.h"),
    "bwd_dq": ("fa_bwd.cu", "ptx.cuh", "fa_internal.h"),
}


def kernel_source_hash(kernel: str) -> str:
    """Short SHA-256 of the code of the CUDA sources `kernel` is built from:
    // comments and blank lines are left out, so that editing a comment does
    not make a traffic capture stale (the sources hold no block comments and
    no string containing //)."""
    return code_digest(os.path.join(ROOT, "tiled_attention_07_gb300", "csrc", name) for name in KERNEL_SOURCES[kernel])


def code_digest(paths) -> str:
    """Short SHA-256 of the given files' lines with // comments and blank
    lines left out."""
    import hashlib

    h = hashlib.sha256()
    for path in paths:
        with open(path, encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (a line ``traffic_bytes_per_launch <kernel> <bytes> <source-hash>``), or
    None if there is none or the kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and parts[0] == "traffic_bytes_per_launch" and parts[1] == kernel:
                    return float(parts[2]) if parts[3] == kernel_source_hash(kernel) else None
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def per_kernel_flops(w):
    """Algorithmic FLOPs per launch of each kernel (GEMMs the kernel performs)."""
    pd = w.pairs() * w.d
    return {"fwd": 4.0 * pd, "bwd_pre": 0.0, "bwd_dkdv": 8.0 * pd, "bwd_dq": 6.0 * pd}


def pick_workload(args):
    import dataclasses

    from tiled_attention_07_gb300 import workloads as W

    w = W.WORKLOADS[args.workload or W.BENCH_WORKLOAD]
    if args.batch is not None and args.batch != w.B:
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_b{args.batch}")
    return w


def run_ours(args):
    import torch

    from tiled_attention_07_gb300 import fa
    from tiled_attention_07_gb300 import workloads as W

    rank, world = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = pick_workload(args)
    host = W.make_inputs(w, device="cpu", with_grad_output=True)
    x = {k: t.to(dev) for k, t in host.items()}
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o = torch.empty_like(q)
    lse = torch.empty(fa.lse_shape(q), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B, H, Nq, d = fa._dims(q)
    Nk = fa._dims(k)[2]
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, Nq, Nk, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = ("fwd", "bwd_pre", "bwd_dkdv", "bwd_dq")

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, w.sm_scale, w.causal, stream)
        if ev is not None:
            ev[1].record(stream)
        for i, phase in enumerate((fa.FA_BWD_PREPROCESS, fa.FA_BWD_DKDV, fa.FA_BWD_DQ)):
            fa.fa_bwd_phase(phase, q, k, v, o, do, lse, dq, dk, dv, w.sm_scale, w.causal, ws, stream)
            if ev is not None:
                ev[2 + i].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    rc, detail = fa.fa_last_device_error(stream)
    if rc != fa.FA_OK:
        raise RuntimeError(f"device error after warm-up: {detail:#x}")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for i in range(K):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop() if clocks else None
    rc, detail = fa.fa_last_device_error(stream)
    if rc != fa.FA_OK:
        raise RuntimeError(f"device error in the timed region: {detail:#x}")

    ms = reduce_max(t0.elapsed_time(t1), dev)
    ms_step = ms / K
    step_flops = w.fwd_flops() + w.bwd_flops()
    value = world * K * step_flops / (ms / 1e3) / 1e12
    kern_ms = {n: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K for j, n in enumerate(names)}
    peaks, peak_src = load_peaks()
    peak, peak_note = tensor_peak(peaks, peak_src, clk)
    kflops = per_kernel_flops(w)
    kernels = {}
    for n in names:
        entry = {"ms": round(kern_ms[n], 4), "share": round(kern_ms[n] / sum(kern_ms.values()), 4)}
        if kflops[n] > 0:
            entry["tflops"] = round(kflops[n] / (kern_ms[n] / 1e3) / 1e12, 2)
            entry["frac"] = round(entry["tflops"] / peak, 4)
        kernels[n] = entry
    dom = max((n for n in names if kflops[n] > 0), key=lambda n: kern_ms[n])
    achieved = kflops[dom] / (kern_ms[dom] / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": committed_traffic(dom), "peak_source": peak_note,
                "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4)}
    fwd_tf = w.fwd_flops() / (kern_ms["fwd"] / 1e3) / 1e12
    bwd_ms = kern_ms["bwd_pre"] + kern_ms["bwd_dkdv"] + kern_ms["bwd_dq"]
    bwd_tf = w.bwd_flops() / (bwd_ms / 1e3) / 1e12
    passes = {"fwd": {"tflops": round(fwd_tf, 2), "frac_of_peak": round(fwd_tf / peak, 4),
                      "frac_of_nominal": round(fwd_tf / NOMINAL_BF16_TFLOPS, 4)},
              "bwd": {"tflops_credited": round(bwd_tf, 2), "frac_of_peak": round(bwd_tf / peak, 4),
                      "frac_of_nominal": round(bwd_tf / NOMINAL_BF16_TFLOPS, 4)},
              "step": {"tflops": round(value / world, 2), "frac_of_peak": round(value / world / peak, 4),
                       "frac_of_nominal": round(value / world / NOMINAL_BF16_TFLOPS, 4)}}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, host, dev, stream, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, host)
    configs = None
    if rank == 0 and not args.no_configs:
        configs = run_configs(args, dev, peaks, peak_src)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp16",
        "data": "synthetic (seeded N(0,1) q, k, v, dO)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal, "sm_scale": w.sm_scale, "layout": w.layout,
                   "step": "fa_fwd + fa_bwd (preprocess, dK/dV pass, dQ pass)",
                   "flops_per_step": step_flops, "l2": "inputs larger than L2 (each of q, k, v, dO is "
                   f"{q.numel() * 2 / 1e6:.0f} MB > 129 MB)", "parallelism": f"replica x{world}"},
        "roofline": roofline, "kernels": kernels, "passes": passes,
        "clocks": clk, "gpu_launches": 4 * K,
        "e2e": e2e, "cpu_baseline": cpu, "configs": configs,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


#: The forward-only configurations, timed after the step for the 'configs'
#: key: the one-head smoke shape, the cross-attention shape, and the short
#: and long causal d = 64 shapes.
FORWARD_CONFIGS = (
    ("C1", "fp16_h1_n128_d64"),
    ("C2", "fp16_h16_nq1000_nk2500_d80"),
    ("C3", "bf16_b4_h12_n512_d64_causal"),
    ("C4", "bf16_b4_h20_n4096_d64_causal"),
)


#: The backward timed on both backward paths for the 'configs' key: the d = 64
#: long causal shape (the fused path exists at d = 64 only).
BACKWARD_CONFIG = ("C4_bwd", "bf16_b4_h20_n4096_d64_causal")


def time_forward(fwd, stream, steps, warmup, flush):
    """Mean device time (ms) of `fwd()` over `steps` calls, each bracketed by
    CUDA events on `stream`; with `flush` (a buffer larger than L2) written
    between calls, outside the events, so every call starts from a cold L2."""
    import torch

    for _ in range(max(warmup, 3)):
        fwd()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 255)
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def forward_roofline(w, ms, peaks, tensor_peak_tflops, fbytes=None):
    """TFLOP/s and GB/s of the algorithmic work of one forward of `w` in `ms`,
    and its fraction of the roofline that bounds it: HBM when the arithmetic
    intensity lies below the measured ridge (tensor peak / HBM bandwidth),
    the tensor peak otherwise."""
    flops = w.fwd_flops()
    fbytes = w.fwd_bytes() if fbytes is None else fbytes
    tflops = flops / (ms / 1e3) / 1e12
    gbs = fbytes / (ms / 1e3) / 1e9
    hbm = flops / fbytes < tensor_peak_tflops * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return {"tflops": round(tflops, 2), "gbs": round(gbs, 1), "bound": "hbm" if hbm else "tensor",
            "frac": round(gbs / peaks["hbm_gbs"] if hbm else tflops / tensor_peak_tflops, 4),
            "peak": peaks["hbm_gbs"] if hbm else tensor_peak_tflops, "unit": "GB/s" if hbm else "TFLOP/s",
            "intensity_flop_per_byte": round(flops / fbytes, 1)}


def run_configs(args, dev, peaks, peak_src):
    """Forward alone on each forward-only configuration, in this process and
    on this GPU: ms per forward (mean of --config-steps), TFLOP/s, GB/s of the
    algorithmic bytes and the fraction of the bounding roofline; inputs under
    256 MB are made cold by a 256 MB write between forwards.  Next to each,
    the oracle's forward on a bounded sample of the same configuration."""
    import torch

    from tiled_attention_07_gb300 import fa
    from tiled_attention_07_gb300 import workloads as W

    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clocks = ClockSampler()
    clocks.start()
    time.sleep(0.3)
    out = {}
    hosts = {}
    for cid, name in FORWARD_CONFIGS:
        w = W.WORKLOADS[name]
        host = W.make_inputs(w, device="cpu", with_grad_output=False)
        hosts[cid] = host
        x = {k: t.to(dev) for k, t in host.items()}
        o = torch.empty_like(x["q"])
        lse = torch.empty(fa.lse_shape(x["q"]), dtype=torch.float32, device=dev)
        in_bytes = sum(t.numel() * t.element_size() for t in x.values())

        def fwd(x=x, o=o, lse=lse, w=w):
            fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, w.sm_scale, w.causal, stream)

        ms = time_forward(fwd, stream, args.config_steps, 10, flush if in_bytes < (256 << 20) else None)
        rc, detail = fa.fa_last_device_error(stream)
        if rc != fa.FA_OK:
            raise RuntimeError(f"device error in {name}: {detail:#x}")
        out[cid] = {"workload": name, "ms": round(ms, 5), "steps": args.config_steps, "launches": args.config_steps,
                    "l2": "256 MB write between forwards" if in_bytes < (256 << 20) else "inputs larger than L2"}
        out[cid]["_ms"] = ms
        del x, o, lse
    # the d = 64 backward of the long causal shape on both backward paths
    w = W.WORKLOADS[BACKWARD_CONFIG[1]]
    host = W.make_inputs(w, device="cpu", with_grad_output=True)
    x = {k: t.to(dev) for k, t in host.items()}
    o = torch.empty_like(x["q"])
    lse = torch.empty(fa.lse_shape(x["q"]), dtype=torch.float32, device=dev)
    fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, w.sm_scale, w.causal, stream)
    grads = {n: torch.empty_like(x[src]) for n, src in (("dq", "q"), ("dk", "k"), ("dv", "v"))}
    B, H, Nq, d = fa._dims(x["q"])
    bwd = {}
    for path_name, path in (("two_pass", fa.FA_BWD_PATH_TWO_PASS), ("fused", fa.FA_BWD_PATH_FUSED)):
        ws = torch.empty(fa.fa_bwd_workspace_bytes_path(B, H, Nq, Nq, d, path), dtype=torch.uint8, device=dev)

        def run(path=path, ws=ws):
            fa.fa_bwd_ex(path, 0, x["q"], x["k"], x["v"], o, x["do"], lse, grads["dq"], grads["dk"], grads["dv"],
                         w.sm_scale, w.causal, ws, stream)

        ms = time_forward(run, stream, args.config_steps, 10, flush)
        rc, detail = fa.fa_last_device_error(stream)
        if rc != fa.FA_OK:
            raise RuntimeError(f"device error in the {path_name} backward: {detail:#x}")
        bwd[path_name] = {"ms": round(ms, 5), "launches": args.config_steps * 3, "_ms": ms}
        del ws
    del x, o, lse, grads
    clk = clocks.stop()
    tpeak, tnote = tensor_peak(peaks, peak_src, clk)
    for entry in bwd.values():
        tf = w.bwd_flops() / (entry.pop("_ms") / 1e3) / 1e12
        entry.update({"tflops_credited": round(tf, 2), "frac": round(tf / tpeak, 4), "peak": tpeak})
    out[BACKWARD_CONFIG[0]] = {"workload": w.name, "steps": args.config_steps, "l2": "256 MB write between calls",
                               "credit": "10*B*H*N^2*d/2 (five products)", "paths": bwd}
    for cid, name in FORWARD_CONFIGS:
        w = W.WORKLOADS[name]
        ms = out[cid].pop("_ms")
        out[cid].update(forward_roofline(w, ms, peaks, tpeak))
        if not args.no_cpu_baseline:
            out[cid]["cpu_baseline"] = cpu_forward_baseline(w, hosts[cid])
    out["clocks"] = clk
    out["tensor_peak_source"] = tnote
    out["hbm_peak_source"] = f"{peak_src} HBM copy bandwidth"
    return out


def cpu_forward_baseline(w, host):
    """The oracle's forward, as it stands, on head (0, 0) of `w` (the whole
    problem when it has one head)."""
    import oracle.attention as ref

    q, k, v = (_head64(host[n], w.layout, 0, 0) for n in ("q", "k", "v"))
    t = time.perf_counter()
    ref.forward(q, k, v, w.sm_scale, w.causal)
    sec = time.perf_counter() - t
    pairs = w.Nq * w.Nk * (0.5 if w.causal else 1.0)
    return {"value": round(4.0 * pairs * w.d / sec / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(),
            "kind": "oracle", "sample": f"forward of head (0,0) of {w.name} in float64 numpy, {sec:.3f} s"}


def run_fwd_only(args):
    """Forward alone on one of the forward-only workloads, optionally split
    over key ranges (fa_fwd_split).  Inputs smaller than L2 are made cold by
    writing a 256 MB scratch buffer between steps, outside the timed kernels;
    each step is timed with CUDA events around the forward launches only."""
    import torch

    from tiled_attention_07_gb300 import fa
    from tiled_attention_07_gb300 import workloads as W

    rank, world = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = pick_workload(args)
    if args.fp8v:
        x = {k: t.to(dev) for k, t in W.fp8v_inputs(w, device="cpu").items() if k != "v8"}
        q, k, v = x["q"], x["k"], x["vt"]
    else:
        x = {k: t.to(dev) for k, t in W.make_inputs(w, device="cpu", with_grad_output=False).items()}
        q, k, v = x["q"], x["k"], x["v"]
    o = torch.empty_like(q)
    lse = torch.empty(fa.lse_shape(q), dtype=torch.float32, device=dev)
    B, H, Nq, d = fa._dims(q)
    Nk = fa._dims(k)[2]
    n_splits = fa.fa_fwd_split_count(B, H, Nq, Nk, d, w.causal) if args.split == "auto" else int(args.split)
    if args.fp8v and n_splits != 1:
        raise SystemExit("--fp8v runs unsplit")
    nbytes = fa.fa_fwd_split_workspace_bytes(B, H, Nq, d, n_splits)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None

    def fwd():
        if args.fp8v:
            fa.fa_fwd_fp8v(q, k, v, o, lse, w.sm_scale, w.causal, stream,
                           mode=fa.FA_FP8V_LAZY_MAX if args.fp8v_lazy else fa.FA_FP8V_PAGE_STEPS)
        elif n_splits > 1:
            fa.fa_fwd_split(q, k, v, o, lse, w.sm_scale, w.causal, n_splits, ws, stream)
        else:
            fa.fa_fwd(q, k, v, o, lse, w.sm_scale, w.causal, stream)

    for _ in range(max(args.warmup, 3)):
        fwd()
    torch.cuda.synchronize(dev)
    rc, detail = fa.fa_last_device_error(stream)
    if rc != fa.FA_OK:
        raise RuntimeError(f"device error after warm-up: {detail:#x}")
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 255)
        evs[i][0].record(stream)
        fwd()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop() if clocks else None
    rc, detail = fa.fa_last_device_error(stream)
    if rc != fa.FA_OK:
        raise RuntimeError(f"device error in the timed region: {detail:#x}")
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), dev)
    ms_step = ms / K
    flops = w.fwd_flops()
    value = world * flops / (ms_step / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    peak, peak_note = tensor_peak(peaks, peak_src, clk)
    if args.fp8v:
        # Half the FLOPs (S = q k^T) at the 16-bit rate P, half (P V) at the
        # 8-bit rate, taken as 2 P (the nominal fp8 : bf16 ratio): time at
        # peak F/2 (1/P + 1/(2P)), i.e. an effective peak of 4P/3.
        peak = round(peak * 4.0 / 3.0, 1)
        peak_note += " x 4/3: S at the 16-bit rate, PV at 2x (nominal fp8:bf16 ratio)"
    # Bound by arithmetic intensity against the measured ridge: below it the
    # forward is an HBM stream and is reported as GB/s of its algorithmic bytes.
    fbytes = w.fwd_bytes() - (w.Nk * w.d * w.B * w.H if args.fp8v else 0)   # e5m2 V: one byte per element
    gbs = world * fbytes / (ms_step / 1e3) / 1e9
    hbm_bound = flops / fbytes < peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    line = {
        "metric": "attention forward TFLOP/s on 1 GB300 (forward-only configuration)", "value": round(value, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (w.dtype + " q,k,o; e5m2 v,p") if args.fp8v else w.dtype, "data": "synthetic (seeded q, k, v)",
        "config": {"workload": w.name + (("_fp8v_lazy" if args.fp8v_lazy else "_fp8v") if args.fp8v else ""), "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk,
                   "d": w.d, "causal": w.causal, "layout": w.layout, "split": n_splits, "flops_per_step": flops,
                   "l2": "256 MB scratch write between steps" if flush is not None else "inputs larger than L2",
                   "parallelism": f"replica x{world}"},
        "roofline": ({"bound": "hbm", "kernel": "fwd" + ("+merge" if n_splits > 1 else ""),
                      "achieved": round(gbs / world, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": round(gbs / world / peaks["hbm_gbs"], 4), "traffic": None,
                      "peak_source": f"{peak_src} HBM copy bandwidth",
                      "algorithmic_bytes": fbytes, "tflops": round(value / world, 2)}
                     if hbm_bound else
                     {"bound": "tensor", "kernel": "fwd" + ("+merge" if n_splits > 1 else ""),
                      "achieved": round(value / world, 2), "peak": peak, "unit": "TFLOP/s",
                      "frac": round(value / world / peak, 4), "traffic": None,
                      "peak_source": peak_note, "gbs": round(gbs / world, 1)}),
        "clocks": clk, "gpu_launches": K * (2 if n_splits > 1 else 1), "e2e": None, "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_bwd_only(args):
    """The backward alone (fa_bwd_ex, all three launches) of --workload on
    --bwd-path: ms per backward, credited TFLOP/s (five products) and its
    fraction of the tensor peak.  Inputs smaller than 256 MB are made cold by
    a 256 MB write between calls, outside the timed launches."""
    import torch

    from tiled_attention_07_gb300 import fa
    from tiled_attention_07_gb300 import workloads as W

    rank, world = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = pick_workload(args)
    path = {"auto": fa.FA_BWD_PATH_AUTO, "two_pass": fa.FA_BWD_PATH_TWO_PASS, "fused": fa.FA_BWD_PATH_FUSED}[
        args.bwd_path]
    x = {k: t.to(dev) for k, t in W.make_inputs(w, device="cpu", with_grad_output=True).items()}
    stream = torch.cuda.current_stream(dev)
    o = torch.empty_like(x["q"])
    lse = torch.empty(fa.lse_shape(x["q"]), dtype=torch.float32, device=dev)
    fa.fa_fwd(x["q"], x["k"], x["v"], o, lse, w.sm_scale, w.causal, stream)
    g = {n: torch.empty_like(x[src]) for n, src in (("dq", "q"), ("dk", "k"), ("dv", "v"))}
    B, H, Nq, d = fa._dims(x["q"])
    Nk = fa._dims(x["k"])[2]
    ws = torch.empty(max(fa.fa_bwd_workspace_bytes_path(B, H, Nq, Nk, d, path), 16), dtype=torch.uint8, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in x.values())
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None

    def run():
        fa.fa_bwd_ex(path, 0, x["q"], x["k"], x["v"], o, x["do"], lse, g["dq"], g["dk"], g["dv"], w.sm_scale,
                     w.causal, ws, stream)

    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier()
    ms = reduce_max(time_forward(run, stream, args.steps, args.warmup, flush), dev)
    barrier()
    clk = clocks.stop() if clocks else None
    rc, detail = fa.fa_last_device_error(stream)
    if rc != fa.FA_OK:
        raise RuntimeError(f"device error: {detail:#x}")
    peaks, peak_src = load_peaks()
    peak, peak_note = tensor_peak(peaks, peak_src, clk)
    tf = w.bwd_flops() / (ms / 1e3) / 1e12
    line = {
        "metric": "attention backward TFLOP/s (credited: five products) on 1 GB300", "value": round(world * tf, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded q, k, v, dO)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                   "bwd_path": args.bwd_path, "flops_per_step": w.bwd_flops(),
                   "l2": "256 MB scratch write between steps" if flush is not None else "inputs larger than L2",
                   "parallelism": f"replica x{world}"},
        "roofline": {"bound": "tensor", "kernel": "bwd (all launches)", "achieved": round(tf, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4), "traffic": None, "peak_source": peak_note},
        "clocks": clk, "gpu_launches": 3 * args.steps, "e2e": None, "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_softmax(args):
    """fa_softmax_rows on one of the named row-softmax workloads: GB/s of the
    algorithmic bytes (every element read once and written once) against
    the measured HBM copy bandwidth.  Inputs smaller than 256 MB are made
    cold by a scratch write between steps, outside the timed kernels."""
    import torch

    from tiled_attention_07_gb300 import fa
    from tiled_attention_07_gb300 import workloads as W

    rank, world = dist_init("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.SOFTMAX_WORKLOADS[args.softmax]
    x = W.softmax_inputs(w.rows, w.T, w.dtype, w.std, w.seed, device="cuda")
    z = torch.empty_like(x)
    lse = torch.empty(w.rows, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = w.bytes_moved()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if nbytes / 2 < (256 << 20) else None
    for _ in range(max(args.warmup, 3)):
        fa.fa_softmax_rows(x, z, lse, stream)
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler() if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 255)
        evs[i][0].record(stream)
        fa.fa_softmax_rows(x, z, lse, stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop() if clocks else None
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs), dev)
    ms_step = ms / K
    gbs = nbytes / (ms_step / 1e3) / 1e9
    peaks, peak_src = load_peaks()
    peak = peaks["hbm_gbs"]
    line = {
        "metric": "row softmax GB/s (algorithmic bytes) on 1 GB300", "value": round(world * gbs, 1), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0, std^2) logits)",
        "config": {"workload": w.name, "rows": w.rows, "T": w.T, "bytes_per_step": nbytes,
                   "l2": "256 MB scratch write between steps" if flush is not None else "inputs larger than L2",
                   "parallelism": f"replica x{world}"},
        "roofline": {"bound": "hbm", "kernel": "softmax_rows", "achieved": round(gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None,
                     "peak_source": f"{peak_src} copy bandwidth"},
        "clocks": clk, "gpu_launches": K, "e2e": None, "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, w, host, dev, stream, world):
    """Same metric through the public API with host buffers: every step copies
    q, k, v, dO from pinned host memory, runs forward and backward, and copies
    O, LSE, dQ, dK, dV back to pinned host memory.

    The steps are pipelined the way a stream of batches would be: two sets of
    device (and host output) buffers, the host-to-device copies on one stream,
    the kernels on another, the device-to-host copies on a third; step i's
    inputs are copied while step i-1 computes and step i-2's results go back.
    The forward starts once q, k, v are in (dO is still on its way) and O, LSE
    go back while the backward runs.  Events order every reuse of a buffer set.
    The timed region runs from the first copy in to the last copy out, so the
    pipeline's fill and drain are inside it."""
    import torch

    from tiled_attention_07_gb300 import fa

    pin = {k: t.pin_memory() for k, t in host.items()}
    B, H, Nq, d = fa._dims(host["q"])
    Nk = fa._dims(host["k"])[2]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    sets = []
    for _ in range(2):
        dx = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
        outs = {"o": torch.empty_like(dx["q"]),
                "lse": torch.empty(fa.lse_shape(dx["q"]), dtype=torch.float32, device=dev),
                "dq": torch.empty_like(dx["q"]), "dk": torch.empty_like(dx["k"]), "dv": torch.empty_like(dx["v"])}
        sets.append({
            "x": dx, "out": outs,
            "ws": torch.empty(fa.fa_bwd_workspace_bytes(B, H, Nq, Nk, d), dtype=torch.uint8, device=dev),
            "hout": {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs.items()},
            "ev_in_fwd": torch.cuda.Event(), "ev_in": torch.cuda.Event(), "ev_fwd": torch.cuda.Event(),
            "ev_cmp": torch.cuda.Event(), "ev_out": torch.cuda.Event(), "used": False,
        })

    def step(i):
        S = sets[i % 2]
        x, out = S["x"], S["out"]
        if S["used"]:
            s_in.wait_event(S["ev_cmp"])      # step i-2's kernels are done with these inputs
        with torch.cuda.stream(s_in):
            for n in ("q", "k", "v"):
                x[n].copy_(pin[n], non_blocking=True)
            S["ev_in_fwd"].record(s_in)       # the forward needs no dO
            x["do"].copy_(pin["do"], non_blocking=True)
            S["ev_in"].record(s_in)
        stream.wait_event(S["ev_in_fwd"])
        if S["used"]:
            stream.wait_event(S["ev_out"])    # step i-2's results have left these outputs
        fa.fa_fwd(x["q"], x["k"], x["v"], out["o"], out["lse"], w.sm_scale, w.causal, stream)
        S["ev_fwd"].record(stream)
        stream.wait_event(S["ev_in"])
        fa.fa_bwd(x["q"], x["k"], x["v"], out["o"], x["do"], out["lse"], out["dq"], out["dk"], out["dv"],
                  w.sm_scale, w.causal, S["ws"], stream)
        S["ev_cmp"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(S["ev_fwd"])     # O and LSE go back while the backward runs
            for n in ("o", "lse"):
                S["hout"][n].copy_(out[n], non_blocking=True)
            s_out.wait_event(S["ev_cmp"])
            for n in ("dq", "dk", "dv"):
                S["hout"][n].copy_(out[n], non_blocking=True)
            S["ev_out"].record(s_out)
        S["used"] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    K = max(1, args.e2e_steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    s_in.wait_stream(stream)
    s_in.wait_stream(s_out)
    t0.record(s_in)
    for i in range(K):
        step(i)
    s_out.wait_stream(stream)
    t1.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    ms = reduce_max(t0.elapsed_time(t1), dev)
    value = world * K * (w.fwd_flops() + w.bwd_flops()) / (ms / 1e3) / 1e12
    bi = sum(t.numel() * t.element_size() for t in pin.values())
    bo = sum(t.numel() * t.element_size() for t in sets[0]["hout"].values())
    return {"value": round(value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": K, "ms_per_step": round(ms / K, 3),
            "pipeline": "2 buffer sets; copies in, kernels, copies out on 3 streams"}


# ---------------------------------------------------------------------------
# the float64 CPU oracle (reported baseline)
# ---------------------------------------------------------------------------

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _head64(t, layout, b, h, n=None):
    from tiled_attention_07_gb300 import workloads as W

    m = W.head_view(t, layout, b, h)
    if n is not None:
        m = m[:n]
    return m.double().numpy()


def cpu_baseline(w, host):
    """The oracle, as it stands, on one full (b, h) head of the workload."""
    import oracle.attention as ref

    q, k, v, do = (_head64(host[n], w.layout, 0, 0) for n in ("q", "k", "v", "do"))
    t = time.perf_counter()
    ref.forward(q, k, v, w.sm_scale, w.causal)
    ref.backward(q, k, v, do, w.sm_scale, w.causal)
    sec = time.perf_counter() - t
    pairs = w.Nq * w.Nk * (0.5 if w.causal else 1.0)
    flops = 14.0 * pairs * w.d   # credited fwd (4) + bwd (10) per pair
    return {"value": round(flops / sec / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "sample": f"head (0,0) of {w.name}: full {w.Nq}x{w.Nk} fwd+bwd in float64 numpy, "
                      f"{sec:.2f} s"}


def run_reference(args):
    """The oracle timed on the host cores (rank 0 only); each step is the
    forward + backward of the top-left 2048 x 2048 block of one head (the
    exact causal sub-problem of its first 2048 queries), heads in turn."""
    rank, world = dist_init("gloo")
    if rank != 0:
        return
    import oracle.attention as ref
    from tiled_attention_07_gb300 import workloads as W

    w = pick_workload(args)
    host = W.make_inputs(w, device="cpu", with_grad_output=True)
    n = min(2048, w.Nq, w.Nk)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def step(i):
        b, h = heads[i % len(heads)]
        q, k, v, do = (_head64(host[m], w.layout, b, h, n) for m in ("q", "k", "v", "do"))
        ref.forward(q, k, v, w.sm_scale, w.causal)
        ref.backward(q, k, v, do, w.sm_scale, w.causal)

    for i in range(max(args.warmup, 3)):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(i)
    sec = time.perf_counter() - t
    pairs = n * n * (0.5 if w.causal else 1.0)
    flops = 14.0 * pairs * w.d
    value = args.steps * flops / sec / 1e12
    sample = f"per step: top-left {n}x{n} causal block of one head of {w.name}, fwd+bwd in float64 numpy"
    line = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(sec / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) q, k, v, dO)", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": w.causal},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.source_hash:
        print(kernel_source_hash(args.source_hash))
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.fwd_only:
        run_fwd_only(args)
    elif args.bwd_only:
        run_bwd_only(args)
    elif args.softmax:
        run_softmax(args)
    else:
        run_ours(args)
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
