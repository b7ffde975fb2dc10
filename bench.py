#!/usr/bin/env python3
"""Benchmark of the PowerSGD compression step on one GB300 (per rank).

A step is one pass of the whole compression over the ResNet-18-shaped
workload (21 conv/fc gradient matrices + 41 vectors, 11.17 M parameters per
worker, W = 4 simulated workers, rank 2): error feedback, P = sum M_w Q,
Gram-Schmidt, Q_w = M_w^T Phat, Qbar, the decompressed update and the new
error buffers, all in the library's step kernel.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own
replica of the workload (weak scaling; the method has no data exchange
between the simulated workers of one GPU and the GPUs).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config c2]
                  [--momentum | --unbiased | --rtopk [--rtopk-top-div D] [--rtopk-sample-div S]]

Configs: c1 (256 x 128), c2 (the ResNet-18 set, default), c3 (LSTM-650),
c4 (the 1.2 B-parameter transformer set), c5r<r> (one 8192 x 8192 layer, W = 8,
rank r), c5s<r> (the same signal on 4096 x 4096, W = 4: a case small enough
for a full ncu capture), c2x<k> (the ResNet-18 set repeated k times).
--momentum fuses the momentum-SGD update into the decompress phase;
--unbiased times the unbiased rank-r variant; --rtopk times rTop-k
sparsification (its four kernels fill the phase slots, and pass 0 is the
roofline kernel).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "gradient GB/s compressed per PowerSGD step (1 GB300) and % of HBM roofline"
UNIT = "GB/s"

# DRAM bytes (read + write) of one launch of the roofline kernel per workload,
# from a one-kernel ncu capture, valid only for the kernel sources whose hash
# (of their code, comments left out) is recorded with it.
NCU_TRAFFIC = {  # {(config, variant): (sources_sha256_prefix, bytes_per_launch)}
    # ResNet-18 set, r = 2, W = 4: ncu capture of two project launches, DRAM
    # 359.5 MB read + 101.0 MB written per launch (the rest of the error write
    # is still in L2 when the kernel ends)
    ("c2", "powersgd"): ("3034e04c68da275f", 460501376),
    # ResNet-18 set, rTop-k, W = 4: ncu capture of two pass-0 launches, DRAM
    # 363.0 MB read + 177.9 MB written per launch
    ("c2", "rtopk"): ("a761099234848755", 540899968),
}


# the sources that define the phase kernels of a step and their launch
# (the allocation-free entry point is not among them; rTop-k adds its own files)
STEP_SOURCES = ("psgd_api.cu", "psgd_cluster.cuh", "psgd_dispatch.h", "psgd_fused.cuh", "psgd_internal.h",
                "psgd_kernels.cuh", "psgd_mma.cuh", "psgd_plan.h", "psgd_umma.cuh",
                "psgd_step_impl.cuh", "psgd_step_r1.cu", "psgd_step_r2.cu", "psgd_step_r4.cu", "psgd_step_r8.cu",
                "psgd_step_r16.cu", "psgd_step_r32.cu")
RTOPK_SOURCES = ("psgd_rtopk.cu", "psgd_rtopk.h")  # and STEP_SOURCES (the API and shared headers)


def _code_only(text: str) -> str:
    """A C++/CUDA source without its comments and blank lines, so that an edit
    of comments alone keeps the recorded counters valid."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_hash(rtopk: bool = False) -> str:
    csrc = os.path.join(ROOT, "rank_gradient_compression_layer_gb300", "csrc")
    h = hashlib.sha256()
    for f in STEP_SOURCES + (RTOPK_SOURCES if rtopk else ()):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def config_of(name: str) -> workloads.Workload:
    if name.startswith("c5r"):
        return workloads.c5_rank_sweep(int(name[3:]))
    if name.startswith("c5s"):  # the rank sweep shrunk to 4096 x 4096, W = 4: a case small enough for ncu
        r = int(name[3:])
        return workloads.scaled(workloads.c5_rank_sweep(r), [(4096, 4096)], name=f"square4096_r{r}_w4", workers=4)
    if name.startswith("c2x"):  # the ResNet-18 set repeated k times (a larger model of the same shapes)
        base = workloads.c2_resnet18()
        return workloads.scaled(base, list(base.layers) * int(name[3:]), name=f"resnet18x{name[3:]}_r2_w4")
    return workloads.ALL[name]()


def project_kernel_name(rp: int) -> str:
    """The project phase's kernel at padded rank rp (PowerSGD, two passes)."""
    return "p1m_kernel" if rp >= 16 else ("p1t_kernel" if rp >= 8 else "p1_kernel")


def algorithmic_bytes(cfg: workloads.Workload, with_update: bool, momentum: bool = False) -> dict:
    """Minimum HBM bytes of one step.

    Per matrix: every worker's gradient is read, its error buffer read and
    written (3 n m floats per worker), plus the factors Phat (n r) and Qbar
    (m r) written; with an update, U (n m) written once; with the fused
    momentum update instead, params and momentum read and written (4 n m).
    Per vector: W reads, plus one write (update) or two reads and two writes
    (momentum update).
    """
    W, r = cfg.workers, cfg.rank
    core = sum(W * 3 * n * m * 4 + 4 * (n + m) * r for n, m in cfg.matrices)
    per = 4 if momentum else (1 if with_update else 0)
    upd = sum(4 * per * n * m for n, m in cfg.matrices)
    vec = sum(4 * (W + per) * n for n, _ in cfg.vectors) if per else 0
    return {"core": core, "update": upd, "vectors": vec, "total": core + upd + vec}


def rtopk_bytes(cfg: workloads.Workload, top_div: int, sample_div: int) -> dict:
    """Minimum HBM bytes of one rTop-k step.

    Per matrix: every worker's gradient read and its error buffer read and
    written (3 n m floats per worker), U written (n m), and each worker's
    message (k indices and k values).  Pass 0 moves all of it but the
    messages; the per-vector terms are as for PowerSGD.
    """
    W = cfg.workers
    pass0 = sum((3 * W + 1) * n * m * 4 for n, m in cfg.matrices)
    msgs = 0
    for n, m in cfg.matrices:
        r = -(-(n * m) // top_div)
        msgs += W * 2 * (-(-r // sample_div)) * 4
    vec = sum(4 * (W + 1) * n for n, _ in cfg.vectors)
    return {"pass0": pass0, "messages": msgs, "vectors": vec, "total": pass0 + msgs + vec}


def unbiased_bytes(cfg: workloads.Workload) -> dict:
    """Minimum HBM bytes of one step of the unbiased variant: every worker's
    gradient read once, P (n r) written, U (n m) written; vectors as above."""
    W, r = cfg.workers, cfg.rank
    core = sum(W * n * m * 4 + 4 * n * r for n, m in cfg.matrices)
    upd = sum(4 * n * m for n, m in cfg.matrices)
    vec = sum(4 * (W + 1) * n for n, _ in cfg.vectors)
    return {"core": core, "update": upd, "vectors": vec, "total": core + upd + vec}


def compressed_bytes(cfg: workloads.Workload) -> int:
    """Gradient bytes compressed per step: W x sum n m x 4."""
    return cfg.workers * sum(n * m for n, m in cfg.matrices) * 4


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="psgd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(name)
        loaded = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# distributed plumbing (timing only; no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_throughput(comp_bytes: float, steps: int, local_ms: float, ws: int, device=None):
    """(ms per step, whole-job GB/s) of ws replicas that each compressed
    comp_bytes per step: the job lasts as long as its slowest rank."""
    total_ms = max_over_ranks(local_ms, ws, device)
    ms_per_step = total_ms / steps
    return ms_per_step, comp_bytes * ws / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------

def time_oracle(cfg: workloads.Workload, steps: int, warmup: int, budget_s: float) -> dict:
    """Times the float64 oracle on this host.  Each step runs on a bounded
    sample of the workload's matrix layers (the largest prefix of the layer
    list, in order, whose step fits the budget share), scaled to GB/s by the
    bytes it compressed."""
    from oracle import powersgd as O

    layers_all = list(cfg.layers)
    mats = [i for i, (n, m) in enumerate(layers_all) if m]
    sig = {}
    st = O.OracleState(layers_all, cfg.rank, cfg.workers, cfg.seed)
    grads = workloads.gradients(cfg, 0, sig)
    # size the sample: probe one full step
    t0 = time.perf_counter()
    st.step(grads, layers=mats)
    full = time.perf_counter() - t0
    per_step = budget_s / max(1, steps + warmup)
    if full <= per_step:
        sample = mats
    else:
        frac = per_step / full
        tot = sum(layers_all[i][0] * layers_all[i][1] for i in mats)
        sample, acc = [], 0
        for i in mats:
            if acc + layers_all[i][0] * layers_all[i][1] > frac * tot and sample:
                break
            sample.append(i)
            acc += layers_all[i][0] * layers_all[i][1]
    el = sum(layers_all[i][0] * layers_all[i][1] for i in sample)
    for _ in range(warmup):
        st.step(grads, layers=sample)
    wall0, cpu0 = time.perf_counter(), time.process_time()
    for _ in range(steps):
        st.step(grads, layers=sample)
    wall = time.perf_counter() - wall0
    cpu = time.process_time() - cpu0
    gbs = cfg.workers * el * 4 * steps / wall / 1e9
    return {"value": gbs, "unit": UNIT, "cores": max(1, round(cpu / wall)), "kind": "oracle",
            "host_cpus": os.cpu_count(), "ms_per_step": wall / steps * 1e3,
            "sample": f"{len(sample)} of {len(mats)} matrix layers ({el} of {cfg.matrix_elements()} elements "
                      f"per worker), W={cfg.workers}, r={cfg.rank}, float64 numpy, {steps} steps"}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def workload_desc(cfg: workloads.Workload) -> str:
    return (f"{cfg.name}: {len(cfg.matrices)} matrices + {len(cfg.vectors)} vectors, "
            f"{cfg.matrix_elements() + cfg.vector_elements()} params per worker, W={cfg.workers}, r={cfg.rank}")


def fill_gradients(ctx, cfg, sets: int, device):
    """`sets` rotating sets of W packed gradient buffers, generated on the device."""
    import torch

    out = []
    for s in range(sets):
        bufs = []
        for w in range(cfg.workers):
            buf = ctx.empty_buffer()
            for li, (n, m) in enumerate(cfg.layers):
                view = ctx.layer_view(buf, li)
                if m:
                    view.copy_(workloads.device_gradient_matrix(cfg, li, s, w, device))
                else:
                    g = torch.Generator(device=device)
                    g.manual_seed(cfg.seed * 7777 + li * 31 + s * 7 + w)
                    view.normal_(0.0, 1.0, generator=g)
            bufs.append(buf)
        out.append(bufs)
    torch.cuda.synchronize()
    return out


def run_ours(args, ws, rank, local):
    import torch

    from rank_gradient_compression_layer_gb300 import PowerSGD

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    cfg = config_of(args.config)
    stream = torch.cuda.Stream(device=device)
    ctx = PowerSGD(cfg.layers, cfg.rank, cfg.workers, seed=cfg.seed, stream=stream, timing=True,
                   unbiased=args.unbiased, compressor="rtopk" if args.rtopk else "powersgd",
                   top_div=args.rtopk_top_div, sample_div=args.rtopk_sample_div,
                   fused=args.fused, queue_lag_kb=args.queue_lag_kb, project_rows=args.project_rows,
                   one_pass=args.one_pass)
    sets = 3
    grads = fill_gradients(ctx, cfg, sets, device)
    upd = ctx.empty_buffer()
    if args.momentum:
        # the fused momentum-SGD update replaces the update write
        params, mom = ctx.empty_buffer(), ctx.empty_buffer()
        params.zero_()
        mom.zero_()

        def one_step(g):
            ctx.step_momentum(g, params, mom, 1e-3, 0.9)
    else:
        def one_step(g):
            ctx.step(g, upd)
    if args.rtopk:
        ab = rtopk_bytes(cfg, args.rtopk_top_div, args.rtopk_sample_div)
    elif args.unbiased:
        ab = unbiased_bytes(cfg)
    else:
        ab = algorithmic_bytes(cfg, with_update=True, momentum=args.momentum)
    comp = compressed_bytes(cfg)
    st = ctx.stats()

    # warm-up; the timed steps run without per-phase events, so the phase
    # kernels' launches overlap (programmatic dependent launch)
    ctx.set_timing(False)
    for i in range(args.warmup):
        one_step(grads[i % sets])
    ctx.sync()
    barrier(ws)
    torch.cuda.synchronize()

    # the timed region: repeats of exactly `steps` steps, each bracketed by a
    # barrier and a device synchronisation, until at least --min-time seconds
    # have passed (so the clock sampler sees the GPU under load); the value
    # is the median repeat, each repeat taking the slowest rank
    sampler = ClockSampler(local)
    sampler.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)

    def timed_repeat() -> float:
        barrier(ws)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            one_step(grads[i % sets])
        ev1.record(stream)
        ctx.sync()
        torch.cuda.synchronize()
        barrier(ws)
        return max_over_ranks(ev0.elapsed_time(ev1), ws, device)

    rep_ms = [timed_repeat()]
    # every rank runs the same number of repeats (from the slowest first one)
    repeats = max(3, int(math.ceil(args.min_time * 1e3 / max(rep_ms[0], 1e-3))))
    repeats = int(max_over_ranks(float(min(repeats, 10000)), ws, device))
    for _ in range(repeats - 1):
        rep_ms.append(timed_repeat())
    clocks = sampler.stop()
    # the same number of steps again with an event between phases: each phase
    # alone, for the per-phase times and the roofline kernel's duration
    ctx.set_timing(True)
    for i in range(args.steps):
        one_step(grads[i % sets])
    ctx.sync()
    phases = ctx.phase_times()  # device ms per phase, averaged over those steps
    med_ms = statistics.median(rep_ms)
    ms_per_step, value = replica_throughput(comp, args.steps, med_ms, 1, device)
    value *= ws  # each repeat is already the max over ranks; ws replicas
    repeat_stats = {"repeats": len(rep_ms), "median_ms_per_step": round(med_ms / args.steps, 5),
                    "min_ms_per_step": round(min(rep_ms) / args.steps, 5),
                    "max_ms_per_step": round(max(rep_ms) / args.steps, 5),
                    "timed_s": round(sum(rep_ms) / 1e3, 3)}
    peaks = measured_peaks()
    if args.rtopk:
        # rTop-k's four phase slots are its kernels; pass 0 moves nearly all the bytes
        phases = dict(zip(("pass0", "pass1", "tail", "apply"), phases.values()))
        project_ms = phases["pass0"]
        project_bytes = ab["pass0"]  # read G, read E, write M of every worker, U zeroed
    elif "step" in phases:
        # the fused step: one launch moves every byte of the step
        project_ms = phases["step"]
        project_bytes = ab["total"]
    else:
        project_ms = phases["project"]
        project_bytes = ab["core"]  # read G, read E, write E of every worker (+ the factors); unbiased: read G
    achieved = project_bytes / (project_ms * 1e-3) / 1e9
    step_achieved = ab["total"] / (ms_per_step * 1e-3) / 1e9
    h = kernel_sources_hash(rtopk=args.rtopk)
    traffic = None
    variant = "rtopk" if args.rtopk else (
        ("powersgd_fused" if st["fused_step"] else ("powersgd_one_pass" if st["one_pass_project"] else "powersgd"))
        if not (args.unbiased or args.momentum) else None)
    if (args.config, variant) in NCU_TRAFFIC and NCU_TRAFFIC[(args.config, variant)][0] == h:
        traffic = NCU_TRAFFIC[(args.config, variant)][1]

    # end to end through the C ABI with host buffers (pinned), copies inside
    e2e = run_e2e(ctx, cfg, args, ws, device)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "parallelism": f"replicas x{ws} (W={cfg.workers} workers "
                   "simulated per GPU)",
                   "l2": "inputs larger than L2: 3 rotating gradient sets of "
                         f"{comp / 1e6:.1f} MB + error buffers {comp / 1e6:.1f} MB per step",
                   "seed": cfg.seed, "out_update": not args.momentum,
                   "fused_momentum_update": bool(args.momentum),
                   "variant": "unbiased" if args.unbiased else (
                       f"rtopk top 1/{args.rtopk_top_div}, sent 1/{args.rtopk_sample_div}" if args.rtopk else
                       "powersgd, one-pass project" if st["one_pass_project"] else "powersgd"),
                   "tile_rows": st["tile_rows"]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "scope": "the dominant kernel alone (the whole step is step_roofline)"
                     if not st["fused_step"] else "the whole step (one fused launch)",
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                     else "fallback 6.8 TB/s",
                     "kernel": ("psgd::rk_pass0_kernel (M = G + E written over E, top digit of |M|, U zeroed)"
                                if args.rtopk else
                                f"psgd::fused_step_kernel<{st['kernel_rank']}> (the whole step: error add, E write, "
                                "P = M Q, Gram-Schmidt, Q_w = M_w^T Phat, Qbar, U)" if st["fused_step"] else
                                f"psgd::p1_kernel<{st['kernel_rank']}> (project: P = G Q)" if args.unbiased else
                                f"psgd::p1c_kernel<{st['kernel_rank']}> (one-pass project on 8-CTA clusters: error "
                                "add, E write, P = M Q, Y_w = M_w^T P)" if st["one_pass_project"] else
                                f"psgd::{project_kernel_name(st['kernel_rank'])}<{st['kernel_rank']}> "
                                "(project: error add, E write, P = M Q)"),
                     "algorithmic_bytes_per_launch": project_bytes, "launch_ms": round(project_ms, 5),
                     "launch_ms_source": "CUDA events around the kernel on the context's stream, "
                                         "averaged over a second pass of the timed steps with per-phase events",
                     "kernel_sources": h},
        "project_fp32": None if st["fused_step"] else project_fp32(cfg, args, project_ms, peaks, device),
        "timing": repeat_stats,
        "step_roofline": {"achieved": round(step_achieved, 1), "frac": round(step_achieved / peaks["hbm_gbs"], 4),
                          "scope": "the whole step: all algorithmic bytes over ms_per_step",
                          "algorithmic_bytes_per_step": ab["total"],
                          "phase_ms": {k: round(v, 5) for k, v in phases.items()}},
        "e2e": e2e,
        "gpu_launches": args.steps * st["launches_per_step"],
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = time_oracle(cfg, steps=3, warmup=1, budget_s=args.cpu_budget)
    ctx.close()
    return out


FP32_LANES_PER_SM = 128  # FP32 FMA lanes per Blackwell SM (nominal)


def project_fp32(cfg, args, project_ms: float, peaks: dict, device):
    """The project kernel's FP32 FMA rate against the CUDA cores' peak.

    Per element and worker the kernel does 2 r FMAs (the error rebuild
    against the previous factors and the projection onto Q); the peak is
    SMs x FP32 lanes x 2 flop x the maximum SM clock.  Not the roofline's
    bound at any rank (HBM is), but it shows how far from arithmetic
    limits the r >= 8 kernels run.
    """
    if args.rtopk or args.unbiased:
        return None
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    flop = 2 * 2 * cfg.rank * cfg.workers * sum(n * m for n, m in cfg.matrices)
    achieved = flop / (project_ms * 1e-3) / 1e12
    peak = sms * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    return {"fma_per_element_worker": 2 * cfg.rank, "achieved_tflops": round(achieved, 2),
            "peak_tflops": round(peak, 1), "frac": round(achieved / peak, 4),
            "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x max SM clock"}


def run_e2e(ctx, cfg, args, ws, device):
    import torch

    host = [torch.empty(ctx.total, dtype=torch.float32).pin_memory() for _ in range(cfg.workers)]
    src = fill_gradients(ctx, cfg, 1, device)[0]
    for w in range(cfg.workers):
        host[w].copy_(src[w].cpu())
    msg = torch.empty(ctx.message_floats, dtype=torch.float32).pin_memory()
    for _ in range(args.warmup):
        ctx.step_host(host, msg)
    steps = max(3, args.steps // 2)
    barrier(ws)
    t0 = time.perf_counter()
    for _ in range(steps):
        ctx.step_host(host, msg)  # waits for its copies
    dt = (time.perf_counter() - t0) / steps
    dt = max_over_ranks(dt, ws, device)
    comp = compressed_bytes(cfg)
    return {"value": round(comp * ws / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": cfg.workers * ctx.total * 4, "d2h_bytes_per_step": ctx.message_floats * 4,
            "ms_per_step": round(dt * 1e3, 4), "steps": steps,
            "api": ("psgd_step_host (pinned host gradients in, sparse messages out)" if args.rtopk else
                    "psgd_step_host (pinned host gradients in, compressed message Phat/Qbar out)")}


def run_reference(args, ws, rank):
    cfg = config_of(args.config)
    if rank != 0:
        return None
    res = time_oracle(cfg, steps=args.steps, warmup=args.warmup, budget_s=args.cpu_budget)
    return {
        "impl": "reference", "metric": METRIC, "value": round(res["value"], 4), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "parallelism": "host cores", "seed": cfg.seed},
        "cpu_baseline": {"value": round(res["value"], 4), "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                         "sample": res["sample"]},
        "e2e": {"value": round(res["value"], 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the reference arm is the float64 CPU oracle (the pages ship no code)",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c2")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for the CPU leg")
    ap.add_argument("--min-time", type=float, default=0.5,
                    help="repeat the timed --steps loop until this many seconds have passed (at least 3 repeats)")
    ap.add_argument("--fused", action="store_true",
                    help="time the fused step (one launch per step over a queue of every phase's tiles, r <= 4)")
    ap.add_argument("--queue-lag-kb", type=int, default=0, help="fused step: queue lag between a layer's phases")
    ap.add_argument("--one-pass", action="store_true",
                    help="time the one-pass project (Y_w = M_w^T P in the project phase; r <= 4)")
    ap.add_argument("--project-rows", type=int, default=0, help="rows per project tile (0: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unbiased", action="store_true",
                    help="time the unbiased rank-r variant (fresh shared Q per step, no error feedback)")
    ap.add_argument("--rtopk", action="store_true", help="time rTop-k sparsification instead of PowerSGD")
    ap.add_argument("--rtopk-top-div", type=int, default=100, help="rTop-k top set: 1 / this of each layer")
    ap.add_argument("--rtopk-sample-div", type=int, default=4, help="rTop-k: 1 / this of the top set is sent")
    ap.add_argument("--momentum", action="store_true",
                    help="time psgd_step_momentum (step + fused momentum-SGD update) instead of psgd_step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, ws, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    out = run_ours(args, ws, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
