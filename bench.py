#!/usr/bin/env python3
"""Benchmark of one paged shared-prefix decode-attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--page-size P]
                    [--layout scatter|contiguous|block128] [--impl reference]

A step is one call of psp_run over the whole synthetic batch: the prefix
kernel of each shared-prefix group (dense or cascade branch, chosen by the
dispatcher) and the split-KV suffix kernel, whose last arriving CTA per
(request, KV head) performs the log-sum-exp merge, with the K/V pool, the
queries and the uploaded plan resident in HBM.  The metric is device time per
step and the achieved HBM bandwidth on the step's unique K/V bytes (a shared
prefix page counts once).  L2 is flushed (a buffer of twice the L2 size is
written and read back) between timed steps, outside the timed events.

The default workload is the largest single-GPU batch: 512 requests sharing a
16,384-token prefix stored once (64 q / 8 KV heads, M_eff 4096, e4m3 K/V
with per-head scales, suffixes U[1,2048], page size 16).  The Llama-shaped
layer without sharing, the 256-request agent batch and the short-prefix batch
are measured in the same process (per_config).

Printed (rank 0, one JSON line): value = unique-KV GB/s over all ranks,
us_per_step, per-kernel times, the dominant kernel's roofline (roofline) and
the other kernels' (roofline_other), the per-request paged comparator (every
request reading the prefix through its own block table) and the read-once
speedup over it, the oracle's CPU baseline, the end-to-end figure through
psp_step_host with host buffers (plan, plan upload, query copy in, output copy
out, every step), the same per-step work as a serving loop that plans the next
step while the device runs the current one (e2e_pipelined), sampled SM clocks, the launch count, a bare read of the same
byte count for context (read_ceiling) and per_config.

--impl reference times the fp64 CPU oracle (the reference arm of this path)
on a bounded sample of the same workload, in the same metric and unit.
Multi-GPU (torchrun): independent replicas, one per GPU, no collective in the
step; value = units of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode-attn µs/step and achieved HBM GB/s (unique KV bytes) vs GB300 peak"
UNIT = "GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the headline workload: the largest single-GPU shared-prefix batch (16,384-token prefix read once,
# M_eff 4096, e4m3 cache); the other workloads are measured beside it in the same process
HEADLINE = "fp8_large"
PER_CONFIG = ("llama8b_noshare", "agent", "short_prefix")
# each kernel's translation unit and the headers it compiles (a recorded DRAM traffic figure
# counts only while all of them are unchanged)
KERNEL_SOURCES = {
    "suffix_splitkv": ("kernel_suffix.cu", "psp_suffix_epi.cuh", "psp_merge.cuh", "psp_device.cuh", "psp_internal.h"),
    "prefix_cascade": ("kernel_prefix_cascade.cu", "psp_merge.cuh", "psp_device.cuh", "psp_internal.h"),
    "prefix_dense": ("kernel_prefix_dense.cu", "psp_sm100.cuh", "psp_merge.cuh", "psp_device.cuh", "psp_internal.h"),
    "expand_kv_indices": ("kernel_merge.cu", "psp_sm100.cuh", "psp_device.cuh", "psp_internal.h"),
}
CSRC = "paged_shared_prefix_gb300/csrc"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--layout", default="scatter", choices=["scatter", "contiguous", "block128"],
                    help="physical page layout of the pool (the generator's layouts)")
    ap.add_argument("--page-size", type=int, default=None)
    ap.add_argument("--impl", default="psp", choices=["psp", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--threshold", type=int, default=0, help="dense/cascade M_eff threshold (0 = built-in)")
    ap.add_argument("--token-flat", action="store_true", help="lower to per-token kv_indices inside the step")
    ap.add_argument("--concurrent", type=int, default=None,
                    help="1: prefix kernels on a side stream concurrent with the suffix kernel, 0: one stream "
                         "(default: the library default for the workload)")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-sharing", action="store_true",
                    help="plan the workload without prefix groups (every request reads its whole context "
                         "through its own block table) and measure that step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads measured beside the headline one")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-ceiling", action="store_true", help="skip the bare-read ceiling measurement")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target oracle CPU time for the baseline")
    ap.add_argument("--sweep-control", action="store_true",
                    help="page size x index layout x footprint control study of the suffix kernel")
    ap.add_argument("--sweep-read-once", action="store_true",
                    help="time the read-once step against the per-request paged step over prefix length x "
                         "members x dtype and report the refit minimum of saved bytes")
    ap.add_argument("--sweep-nested", action="store_true",
                    help="nested prefix groups: both levels read once vs the root alone vs no sharing")
    ap.add_argument("--sweep-nested-read-once", action="store_true",
                    help="nested segments read once or through each block table, over blocks x segment length")
    ap.add_argument("--sweep-threshold", action="store_true",
                    help="time the dense and cascade prefix kernels over an M_eff sweep and report the refit threshold")
    return ap.parse_args()


def peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def describe(case) -> str:
    w = case.workload
    return (f"{w.name}: B={case.batch}, Hq={w.num_q_heads}, Hkv={w.num_kv_heads}, d={w.head_dim}, "
            f"q={w.q_dtype}, kv={w.kv_dtype}, o={w.o_dtype}, shared prefix {w.prefix_len} tokens, "
            f"private U[{w.private_lo},{w.private_hi}], page size {case.page_size}, "
            f"{case.num_pages} pages ({case.layout})")


def src_hash(files) -> str:
    """First 16 hex digits of the SHA-256 of the named csrc files' bytes, in order."""
    h = hashlib.sha256()
    try:
        for name in files:
            with open(os.path.join(ROOT, CSRC, name), "rb") as f:
                h.update(f.read())
    except OSError:
        return ""
    return h.hexdigest()[:16] if files else ""


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(f"{kernel}@{workload}")
    if not ent or ent.get("source_sha256_16") != src_hash(KERNEL_SOURCES.get(kernel, ())):
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- oracle

def oracle_timing(case, target_s: float, seed: int = 0) -> dict:
    """Times the fp64 oracle on a random sample of (request, head) rows and scales the
    measured time by the share of context tokens the sample covers."""
    import oracle
    w = case.workload
    B, Hq = case.batch, w.num_q_heads
    rng = np.random.default_rng(seed)
    order = rng.permutation(B * Hq)
    total_tok = float(case.kv_len.astype(np.int64).sum() * Hq)
    # calibrate on a small sample, then size the real one
    n = min(len(order), max(8, oracle.num_threads()))
    t = time.perf_counter()
    rows = order[:n]
    oracle.attend(case, rows // Hq, rows % Hq)
    dt = time.perf_counter() - t
    tok = float(case.kv_len[rows // Hq].astype(np.int64).sum())
    rate = tok / max(dt, 1e-9)
    n2 = int(min(len(order), max(n, target_s * rate / max(tok / n, 1.0))))
    rows = order[:n2]
    t = time.perf_counter()
    oracle.attend(case, rows // Hq, rows % Hq)
    dt = time.perf_counter() - t
    reps = 1
    if n2 == len(order) and dt < 0.5 * target_s:
        # the whole step is shorter than the target: repeat it and average
        reps = 0
        t = time.perf_counter()
        while reps < 10000 and (reps == 0 or time.perf_counter() - t < target_s):
            oracle.attend(case, rows // Hq, rows % Hq)
            reps += 1
        dt = (time.perf_counter() - t) / reps
    tok = float(case.kv_len[rows // Hq].astype(np.int64).sum())
    step_s = dt * total_tok / tok
    return {"step_s": step_s, "rows": int(n2), "total_rows": int(B * Hq), "cores": oracle.num_threads(),
            "sample_s": dt * reps, "reps": reps}


# ------------------------------------------------------------------ replicas

def aggregate_replicas(ms_local: float, unique_bytes: int, world: int, device=None) -> tuple:
    """Slowest rank's ms per step and the whole-job GB/s: every rank runs its own full
    step (weak scaling), so the job moves world x unique_bytes per slowest step time."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * unique_bytes / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ main

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    case = workloads.make_case(args.workload, args.seed, page_size=args.page_size, layout=args.layout)
    ub = workloads.unique_kv_bytes(case)
    per_step_target = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_timing(case, per_step_target / 4)
    times = [oracle_timing(case, per_step_target, seed=i)["step_s"] for i in range(args.steps)]
    last = oracle_timing(case, per_step_target, seed=args.steps)
    step_s = statistics.mean(times)
    val = ub / step_s / 1e9
    w = case.workload
    out = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "us_per_step": step_s * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(case)},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                         "sample": f"{last['rows']} of {last['total_rows']} (request, head) rows per step, "
                                   f"time scaled by context tokens covered"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))
    return 0


def sweep_threshold(args):
    """Dispatcher refit: with 8 KV heads, time the prefix kernel of both branches over
    prefix length x cache type x batch x GQA group; the refit threshold T (dense iff
    M_eff >= T) is the swept M_eff with the least summed log(time / faster time), reported
    per (cache, prefix) cell and over all points."""
    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    rows = []
    cells = [("bf16", "agent", P) for P in (1024, 4096, 16384)] + [("fp8_e4m3", "fp8_large", P) for P in (1024, 4096, 16384)]
    for cache, base, P in cells:
        for G in (1, 2, 4, 8):
            for B in (4, 8, 16, 32, 64, 128, 256, 512):
                m_eff = B * G
                if m_eff < 16 or m_eff > 4096:
                    continue
                case = workloads.make_case(base, 11, batch=B, prefix_len=P, private_range=(1, 16),
                                           num_q_heads=8 * G, num_kv_heads=8)
                tens = to_device(case, dev)
                o = torch.empty((B, 8 * G, 128), dtype=torch.bfloat16, device=dev)
                res = {}
                for branch, thr in (("dense", 1), ("cascade", 1 << 30)):
                    step = psp.DecodeStep.for_case(case, dense_threshold=thr, read_once_min_tokens=-1,
                                                   read_once_min_mib=-1)
                    step.plan_case(case)
                    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
                    step.upload(ws)
                    step.set_kernel_timing(True)
                    times = []
                    for i in range(8):
                        step.run(tens["q"], tens["k"], tens["v"], o, None, tens["ks"], tens["vs"])
                        torch.cuda.synchronize()
                        if i >= 3:
                            times += [ms for n, ms in step.kernel_times() if n.startswith("prefix")]
                    res[branch] = statistics.median(times) * 1e3
                    step.close()
                rows.append({"cache": cache, "prefix_tokens": P, "G": G, "B": B, "m_eff": m_eff,
                             "dense_us": res["dense"], "cascade_us": res["cascade"]})
    # refit: the swept M_eff whose rule (dense iff M_eff >= T) has the least summed
    # log(time / faster time), per (cache, prefix) cell and over every point
    cands = sorted({r["m_eff"] for r in rows})

    def regret(pts, T):
        return sum(math.log((r["dense_us"] if r["m_eff"] >= T else r["cascade_us"]) /
                            min(r["dense_us"], r["cascade_us"])) for r in pts)
    cell_thr = {}
    for cache, _, P in cells:
        pts = [r for r in rows if r["cache"] == cache and r["prefix_tokens"] == P]
        cell_thr[f"{cache}@{P}"] = min(cands, key=lambda T: (regret(pts, T), T))
    best = min(cands, key=lambda T: (regret(rows, T), T))
    known = {"refit_regret": regret(rows, best), "regret_by_threshold": {T: regret(rows, T) for T in cands}}
    print(json.dumps({"sweep": rows, "cell_thresholds": cell_thr, "refit_threshold": best, **known,
                      "gpu": torch.cuda.get_device_name(0), "kv_heads": 8}))
    return 0


def to_device(case, dev):
    import torch

    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q), k=t(case.k_pool), v=t(case.v_pool), ks=t(case.k_scale), vs=t(case.v_scale))


def make_outputs(case, dev):
    import torch
    w = case.workload
    odt = torch.float32 if w.o_dtype == "f32" else torch.bfloat16
    o = torch.empty((case.batch, w.num_q_heads, w.head_dim), dtype=odt, device=dev)
    lse = torch.empty((case.batch, w.num_q_heads), dtype=torch.float32, device=dev)
    return o, lse


def kernel_roofline(name, ms, case, info, pk, pk_src):
    """Roofline entry of one kernel: algorithmic work per launch / its mean event time."""
    w = case.workload
    Hkv, d = w.num_kv_heads, w.head_dim
    tok_bytes = 2 * Hkv * d * workloads.elem_bytes(w.kv_dtype)
    if name in ("prefix_dense", "prefix_cascade"):
        m_eff = int(case.batch * (w.num_q_heads // Hkv))
        flops = 4.0 * m_eff * info["shared_tokens"] * d * Hkv
        achieved = flops / (ms * 1e-3) / 1e12
        peak = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        note = f"{pk_src} bf16 burst"
        if w.kv_dtype == "fp8_e4m3" and name == "prefix_dense":
            # e4m3 products: the measured bf16 peak times the nominal e4m3 / bf16 ratio (4.5 / 2.25)
            peak *= 2.0
            note = f"{pk_src} bf16 burst x 2 (nominal e4m3 / bf16 ratio)"
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic(name, w.name), "kernel": name, "us": ms * 1e3,
                "algorithmic": f"{flops:.4g} FLOP per launch = 4 x M_eff {m_eff} x {info['shared_tokens']} shared "
                               f"tokens x d {d} x Hkv {Hkv}",
                "peak_source": note}
    if name == "suffix_splitkv":
        alg = info["suffix_tokens"] * tok_bytes
        desc = f"{alg} B per launch = {info['suffix_tokens']} suffix tokens x {tok_bytes} B (K+V, all KV heads)"
    else:
        alg = info["kv_indices_len"] * 4
        desc = f"{alg} B per launch = {info['kv_indices_len']} indices x 4 B written"
    achieved = alg / (ms * 1e-3) / 1e9
    peak = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": recorded_traffic(name, w.name), "kernel": name, "us": ms * 1e3, "algorithmic": desc,
            "peak_source": pk_src}


class Runner:
    """Device state shared by every measurement of one bench process."""

    def __init__(self, dev, stream):
        import torch
        self.dev, self.stream = dev, stream
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
        self.flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(self):
        import torch
        # write a buffer of twice the L2 size (evicts the step's data), then read it back so
        # no dirty line is left whose write-back would land inside the next timed step
        self.flush.fill_(1.0)
        torch.sum(self.flush, dim=0, out=self.sink)

    def time_steps(self, fn, steps, warmup, clocks=None):
        """Mean ms of `steps` calls of fn() (each after an untimed L2 flush), CUDA events on the
        launching stream; returns (ms list, wall seconds of the timed loop)."""
        import torch
        for _ in range(max(3, warmup)):
            self.flush_l2()
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if clocks:
            clocks.start()
        wall0 = time.perf_counter()
        for a, b in evs:
            self.flush_l2()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        return [a.elapsed_time(b) for a, b in evs], wall

    def kernel_times(self, step, run, n):
        """Per-kernel mean ms from psp's own events around each launch (a separate pass: the
        events sit between the kernels and disable the dependent launch)."""
        import torch
        step.set_kernel_timing(True)
        kern = {}
        for _ in range(n):
            self.flush_l2()
            run()
            torch.cuda.synchronize()
            for name, kms in step.kernel_times():
                kern.setdefault(name, []).append(kms)
        step.set_kernel_timing(False)
        return {k: statistics.mean(v) for k, v in kern.items()}


def measure_case(psp, runner, case, steps, warmup, *, threshold=0, token_flat=False, concurrent=False,
                 comparator=True, clocks=None, tensors=None, read_once=None):
    """One workload: whole-step times, per-kernel times, plan facts and the per-request paged
    comparator (the same batch with every request reading its prefix through its own table)."""
    import torch
    dev, stream = runner.dev, runner.stream
    tens = tensors or to_device(case, dev)
    o, lse = make_outputs(case, dev)
    step = psp.DecodeStep.for_case(case, dense_threshold=threshold, token_flat=token_flat, concurrent=concurrent,
                                   **(read_once or {}))
    t_plan = []
    for _ in range(5):
        t0 = time.perf_counter()
        step.plan_case(case)
        t_plan.append(time.perf_counter() - t0)
    info = step.plan_info()
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
    step.upload(ws, stream)

    def run():
        step.run(tens["q"], tens["k"], tens["v"], o, lse, tens["ks"], tens["vs"], stream)

    ms_list, wall = runner.time_steps(run, steps, warmup, clocks)
    n_kernel_steps = max(3, min(steps, 20))
    kern = runner.kernel_times(step, run, n_kernel_steps)
    ub = workloads.unique_kv_bytes(case)
    ms = statistics.mean(ms_list)
    names = {0: "none", 1: "cascade", 2: "dense", 3: "paged"}
    info["branches"] = [names[int(b)] for b in step.plan_query("group_branch")] if case.num_groups else []
    res = {"case": case, "step": step, "ws": ws, "tens": tens, "o": o, "lse": lse, "info": info,
           "ms": ms, "ms_list": ms_list, "wall": wall, "kernels_ms": kern, "plan_us": statistics.median(t_plan) * 1e6,
           "unique_bytes": ub, "paged_bytes": workloads.paged_kv_bytes(case),
           "launches_per_step": len(kern)}
    if comparator and case.num_groups > 0:
        nc = case.without_sharing()
        cstep = psp.DecodeStep.for_case(nc, token_flat=token_flat)
        cstep.plan_case(nc)
        cws = torch.empty(cstep.workspace_size(), dtype=torch.uint8, device=dev)
        cstep.upload(cws, stream)
        cms, _ = runner.time_steps(
            lambda: cstep.run(tens["q"], tens["k"], tens["v"], o, lse, tens["ks"], tens["vs"], stream),
            max(5, min(steps, 20)), 3)
        cmean = statistics.mean(cms)
        res["paged_comparator"] = {"us_per_step": cmean * 1e3, "speedup_read_once": cmean / ms,
                                   "bytes_per_step": workloads.paged_kv_bytes(case),
                                   "what": "the same batch planned without prefix groups: every request reads "
                                           "the shared prefix through its own block table (suffix kernel only)"}
        cstep.close()
        del cws
    return res


def e2e_pipelined(psp, step, case, tens, ws, stream, steps, warmup):
    """Serving loop through the C ABI with host buffers: every step copies its queries in from
    pinned memory, plans (psp_plan), uploads the plan (psp_upload), runs (psp_run) and copies
    its output and LSE back into pinned memory.  The host plans step i + 1 while the device
    runs step i and waits for step i's output one step later; queries and outputs are
    double-buffered on the device and the two copy directions run on streams of their own.
    L2 is not flushed: the step's K/V bytes are several times the L2 size.  Returns
    (seconds per step, H2D bytes per step, D2H bytes per step)."""
    import torch
    w = case.workload
    dev = tens["k"].device
    qh = torch.from_numpy(np.ascontiguousarray(case.q).view(np.int16 if w.q_dtype == "bf16" else np.float32))
    qh = qh.pin_memory()
    qd, od, ld, oh, lh = [], [], [], [], []
    for _ in range(2):
        qd.append(torch.empty_like(tens["q"]))
        o, lse = make_outputs(case, dev)
        od.append(o)
        ld.append(lse)
        oh.append(torch.empty(o.shape, dtype=torch.int16 if w.o_dtype == "bf16" else torch.float32).pin_memory())
        lh.append(torch.empty(lse.shape, dtype=torch.float32).pin_memory())
    batch, keep = step.make_case_batch(case)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ring = 4
    ev_q = [torch.cuda.Event() for _ in range(ring)]
    ev_run = [torch.cuda.Event() for _ in range(ring)]
    ev_o = [torch.cuda.Event() for _ in range(ring)]

    def one(i):
        k = i % 2
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(ev_run[(i - 2) % ring])   # step i - 2 has read this query buffer
            qd[k].view(qh.dtype).copy_(qh, non_blocking=True)
            ev_q[i % ring].record(h2d)
        step.plan_batch(batch)
        step.upload(ws, stream)
        stream.wait_event(ev_q[i % ring])
        step.run(qd[k], tens["k"], tens["v"], od[k], ld[k], tens["ks"], tens["vs"], stream)
        ev_run[i % ring].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_run[i % ring])
            oh[k].copy_(od[k].view(oh[k].dtype), non_blocking=True)
            lh[k].copy_(ld[k], non_blocking=True)
            ev_o[i % ring].record(d2h)
        if i >= 1:
            ev_o[(i - 1) % ring].synchronize()           # step i - 1's output is on the host

    for i in range(max(3, warmup)):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    per_step = (time.perf_counter() - t0) / steps
    plan_bytes = sum(int(step.plan_query(f).nbytes) for f in psp.FIELDS)
    h2d_bytes = int(qh.numel() * qh.element_size()) + plan_bytes
    d2h_bytes = int(oh[0].numel() * oh[0].element_size() + lh[0].numel() * 4)
    del keep
    return per_step, h2d_bytes, d2h_bytes


def config_summary(res, pk, pk_src):
    case, info = res["case"], res["info"]
    ub, ms = res["unique_bytes"], res["ms"]
    gbs = ub / (ms * 1e-3) / 1e9
    out = {"workload": describe(case), "us_per_step": ms * 1e3, "unique_kv_bytes": ub, "value": gbs, "unit": UNIT,
           "hbm_frac_of_8tbs": gbs / 8000.0, "frac_of_measured_hbm": gbs / pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
           "kernels_us": {k: v * 1e3 for k, v in res["kernels_ms"].items()},
           "kernel_rooflines": {k: kernel_roofline(k, v, case, info, pk, pk_src) for k, v in res["kernels_ms"].items()},
           "plan": {k: info[k] for k in ("num_splits", "num_chunks", "suffix_ctas", "prefix_dense_ctas",
                                          "prefix_cascade_ctas", "dense_threshold", "branches")}}
    if "paged_comparator" in res:
        out["paged_comparator"] = {k: v for k, v in res["paged_comparator"].items() if k != "what"}
    return out


def sweep_read_once(args):
    """Dispatcher refit of the read-once choice: for prefix lengths x members x cache dtype,
    the step with the prefix read once (prefix kernel + suffix kernel) against the same batch
    planned without groups (every member reads the prefix through its own block table).
    Reports the bytes that reading once saves, (members - 1) x shared tokens x bytes per
    token, and the speedup; the refit minimum is the smallest saved size from which reading
    once is never slower."""
    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    runner = Runner(dev, torch.cuda.current_stream(dev))
    rows = []
    for name, heads in (("short_prefix", 16), ("agent", 32), ("fp8_large", 64)):
        for P in (128, 256, 512, 1024, 2048, 4096):
            for B in (8, 32, 128, 256):
                case = workloads.make_case(name, 13, batch=B, prefix_len=P, private_range=(256, 2048),
                                           num_q_heads=heads, num_kv_heads=8)
                r = measure_case(psp, runner, case, 10, 3)
                tb = case.kv_token_bytes()
                rows.append({"workload": name, "kv_dtype": case.workload.kv_dtype, "prefix": P, "members": B,
                             "m_eff": B * heads // 8, "saved_bytes": (B - 1) * P * tb,
                             "read_once_us": r["ms"] * 1e3, "paged_us": r["paged_comparator"]["us_per_step"],
                             "speedup": r["paged_comparator"]["speedup_read_once"]})
                r["step"].close()
                del r
    rows.sort(key=lambda x: x["saved_bytes"])
    floor = None
    for i, x in enumerate(rows):
        if all(y["speedup"] >= 1.0 for y in rows[i:]):
            floor = x["saved_bytes"]
            break
    print(json.dumps({"sweep": rows, "refit_min_saved_bytes": floor, "gpu": torch.cuda.get_device_name(0)}))
    return 0


def sweep_nested(args):
    """Nested prefix groups ("Track C Document 10": a radix tree of shared beginnings; sharing
    per user on top of what every user shares): 256 requests share a 4096-token root prefix,
    and each block of 256 / n requests shares one more segment on top of it, then private
    suffixes U[128, 1024].  Three plans of the same batch and pool: both levels read once
    (nested groups), the root alone read once (each request reads its block's segment through
    its own block table), and no sharing.  bf16 (32 / 8 heads) and e4m3 (64 / 8 heads)."""
    import dataclasses

    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    runner = Runner(dev, torch.cuda.current_stream(dev))
    rows = []
    for name in ("agent", "fp8_large"):
        for n_sub, seg in ((4, 2048), (16, 2048), (16, 8192), (16, 512), (64, 1024)):
            case = workloads.make_case(name, 17, batch=256, prefix_len=4096, private_range=(128, 1024),
                                       nested=(n_sub, seg))
            nested = measure_case(psp, runner, case, args.steps, args.warmup)
            root = dataclasses.replace(case, prefix_group=np.zeros(case.batch, np.int32),
                                       group_prefix_len=case.group_prefix_len[:1].copy(), group_parent=None)
            alone = measure_case(psp, runner, root, args.steps, args.warmup, comparator=False,
                                 tensors=nested["tens"])
            # every segment read once, whatever the dispatcher's read-once minimums say
            forced = measure_case(psp, runner, case, args.steps, args.warmup, comparator=False,
                                  tensors=nested["tens"], read_once=dict(read_once_min_tokens=-1,
                                                                         read_once_min_mib=-1))
            rows.append({"workload": name, "kv_dtype": case.workload.kv_dtype, "batch": case.batch, "root": 4096,
                         "subgroups": n_sub, "segment": seg, "unique_kv_bytes": nested["unique_bytes"],
                         "nested_us": nested["ms"] * 1e3, "root_only_us": alone["ms"] * 1e3,
                         "no_sharing_us": nested["paged_comparator"]["us_per_step"],
                         "speedup_vs_root_only": alone["ms"] / nested["ms"],
                         "speedup_vs_no_sharing": nested["paged_comparator"]["speedup_read_once"],
                         "nested_gbs": nested["unique_bytes"] / (nested["ms"] * 1e-3) / 1e9,
                         "branches": nested["info"]["branches"][:2], "kernels_us":
                             {k: v * 1e3 for k, v in nested["kernels_ms"].items()},
                         "all_read_once_us": forced["ms"] * 1e3, "all_read_once_branches": forced["info"]["branches"][:2],
                         "all_read_once_kernels_us": {k: v * 1e3 for k, v in forced["kernels_ms"].items()}})
            for r in (nested, alone, forced):
                r["step"].close()
            del nested, alone, forced
    print(json.dumps({"sweep_nested": rows, "gpu": torch.cuda.get_device_name(0)}))
    return 0


def sweep_nested_read_once(args):
    """Read-once choice for nested segments: 256 requests under a 4096-token root read once, n
    blocks each sharing an S-token segment, suffixes U[128, 1024]; the step with every segment
    read once against the same batch with the segments read through each request's block table
    (the root alone shared), over n x S and both caches.  Reports the bytes a segment saves when
    read once, (members - 1) x S x bytes per token, and the speedup."""
    import dataclasses

    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    runner = Runner(dev, torch.cuda.current_stream(dev))
    rows = []
    always = dict(read_once_min_tokens=-1, read_once_min_mib=-1)
    for name in ("agent", "fp8_large"):
        for n_sub in (4, 16, 64):
            for seg in (256, 512, 1024, 2048, 4096):
                case = workloads.make_case(name, 19, batch=256, prefix_len=4096, private_range=(128, 1024),
                                           nested=(n_sub, seg))
                once = measure_case(psp, runner, case, args.steps, args.warmup, comparator=False, read_once=always)
                root = dataclasses.replace(case, prefix_group=np.zeros(case.batch, np.int32),
                                           group_prefix_len=case.group_prefix_len[:1].copy(), group_parent=None)
                paged = measure_case(psp, runner, root, args.steps, args.warmup, comparator=False,
                                     tensors=once["tens"], read_once=always)
                members = case.batch // n_sub
                rows.append({"workload": name, "kv_dtype": case.workload.kv_dtype, "subgroups": n_sub, "segment": seg,
                             "members": members, "m_eff": members * (case.workload.num_q_heads // 8),
                             "saved_bytes": (members - 1) * seg * case.kv_token_bytes(),
                             "read_once_us": once["ms"] * 1e3, "paged_us": paged["ms"] * 1e3,
                             "speedup": paged["ms"] / once["ms"]})
                for r in (once, paged):
                    r["step"].close()
                del once, paged
    print(json.dumps({"sweep_nested_read_once": rows, "gpu": torch.cuda.get_device_name(0)}))
    return 0


def sweep_control(args):
    """Control study of page size and index contiguity on the suffix kernel ("The 25% Page-Size
    Slowdown That Wasn't", "When source beats intuition": FlashInfer decode moved -1.0..+1.3%
    between contiguous and scattered indices over 0.03-8.59 GB).  Llama-shaped layers (32 / 8
    heads, d = 128, bf16, contexts U[2048, 4096]) of 2 to 680 requests, at page sizes 1 and 16,
    with the pages laid out contiguously, in 128-token blocks or scattered; block tables from
    the seeded generator, K/V filled on the device with N(0, 1) bf16 values (the step's time
    does not depend on the values; the host never holds the larger pools)."""
    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    runner = Runner(dev, stream)
    rows = []
    for B in (2, 6, 24, 96, 384, 680):
        for ps in (1, 16):
            for layout in ("contiguous", "block128", "scatter"):
                case = workloads.make_case("llama8b_noshare", 17, batch=B, page_size=ps, layout=layout,
                                           tables_only=True)
                w = case.workload
                shape = (case.num_pages, ps, w.num_kv_heads, w.head_dim)
                kp = torch.randn(shape, dtype=torch.bfloat16, device=dev)
                vp = torch.randn(shape, dtype=torch.bfloat16, device=dev)
                q = torch.randn((B, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
                o = torch.empty_like(q)
                step = psp.DecodeStep.for_case(case)
                step.plan_case(case)
                ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
                step.upload(ws, stream)
                ms, _ = runner.time_steps(lambda: step.run(q, kp, vp, o, None, None, None, stream), 10, 3)
                ub = workloads.unique_kv_bytes(case)
                us = statistics.median(ms) * 1e3
                rows.append({"requests": B, "page_size": ps, "layout": layout, "kv_bytes": ub,
                             "us_per_step": us, "gbs": ub / (us * 1e-6) / 1e9})
                step.close()
                del kp, vp, ws
                torch.cuda.empty_cache()
    for r in rows:
        base = next(x for x in rows if x["requests"] == r["requests"] and x["page_size"] == r["page_size"]
                    and x["layout"] == "contiguous")
        r["vs_contiguous_pct"] = 100.0 * (r["us_per_step"] / base["us_per_step"] - 1.0)
    print(json.dumps({"control": rows, "gpu": torch.cuda.get_device_name(0)}))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep_threshold:
        return sweep_threshold(args)
    if args.sweep_read_once:
        return sweep_read_once(args)
    if args.sweep_control:
        return sweep_control(args)
    if args.sweep_nested:
        return sweep_nested(args)
    if args.sweep_nested_read_once:
        return sweep_nested_read_once(args)

    import torch
    import torch.distributed as dist

    import paged_shared_prefix_gb300 as psp

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    runner = Runner(dev, stream)
    pk, pk_src = peaks()

    case = workloads.make_case(args.workload, args.seed + rank, page_size=args.page_size, layout=args.layout)
    if args.no_sharing:
        case = case.without_sharing()
    w = case.workload
    concurrent = bool(args.concurrent) if args.concurrent is not None else False
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    head = measure_case(psp, runner, case, args.steps, args.warmup, threshold=args.threshold,
                        token_flat=args.token_flat, concurrent=concurrent, comparator=not args.no_comparator,
                        clocks=clocks)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ub = head["unique_bytes"]
    ms, value = aggregate_replicas(head["ms"], ub, world, dev)
    info, kmean = head["info"], head["kernels_ms"]
    step, ws, tens, o, lse = head["step"], head["ws"], head["tens"], head["o"], head["lse"]

    # ---- single-launch read ceiling: a bare read of as many bytes as the step's unique K/V
    # (torch's sum kernel, L2 flushed the same way), for context beside the roofline peak
    ceil = None
    if not args.no_read_ceiling:
        buf = torch.empty(ub // 4, dtype=torch.float32, device=dev).fill_(1.0)
        cms, _ = runner.time_steps(lambda: torch.sum(buf, dim=0, out=runner.sink), 8, 2)
        ceil = {"gbs": buf.numel() * 4 / (statistics.mean(cms) * 1e-3) / 1e9, "bytes": int(buf.numel() * 4),
                "how": "torch.sum over a float32 buffer of the unique K/V size, one launch, L2 flushed as for the step"}
        del buf

    rooflines = {k: kernel_roofline(k, v, case, info, pk, pk_src) for k, v in kmean.items()}
    order = sorted(kmean, key=kmean.get, reverse=True)
    dom = order[0]
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "f32", "bf16": "bf16", "fp8_e4m3": "fp8_e4m3"}[w.kv_dtype],
        "data": "synthetic",
        "config": {"workload": describe(case), "l2": "flushed between steps (2x L2 buffer written then read back, untimed)",
                   "parallelism": f"replicas x{world}", "token_flat": bool(args.token_flat),
                   "concurrent_prefix": concurrent},
        "unique_kv_bytes": ub, "paged_kv_bytes": head["paged_bytes"],
        "hbm_frac_of_8tbs": value / world / 8000.0,
        "kernels_ms": kmean, "plan_us": head["plan_us"],
        "roofline": rooflines[dom],
        "roofline_other": [rooflines[k] for k in order[1:]],
        "read_ceiling": ceil, "clocks": clk, "gpu_launches": args.steps * head["launches_per_step"],
        "wall_s": head["wall"],
        "plan": {k: info[k] for k in ("num_splits", "num_chunks", "suffix_ctas", "prefix_dense_ctas",
                                       "prefix_cascade_ctas", "dense_threshold", "num_sms", "branches",
                                       "read_once_min_tokens", "read_once_min_mib")},
    }
    if "paged_comparator" in head:
        result["paged_comparator"] = head["paged_comparator"]

    # ---- end to end through the C ABI with host buffers
    if not args.no_e2e:
        qh = torch.from_numpy(np.ascontiguousarray(case.q).view(np.int16 if w.q_dtype == "bf16" else np.float32))
        qh = qh.pin_memory()
        oh = torch.empty(o.shape, dtype=torch.int16 if w.o_dtype == "bf16" else torch.float32).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        qd = torch.empty_like(tens["q"])
        batch, keep = step.make_case_batch(case)
        devt = step.tensors(qd, tens["k"], tens["v"], o, lse, tens["ks"], tens["vs"])
        e2e = []
        for i in range(3 + args.steps):
            runner.flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            step.step_host(batch, qh, oh, lh, devt, ws, stream)
            if i >= 3:
                e2e.append(time.perf_counter() - t0)
        e2e_s = statistics.mean(e2e)
        plan_bytes = sum(int(step.plan_query(f).nbytes) for f in psp.FIELDS)
        result["e2e"] = {"value": world * ub / e2e_s / 1e9, "unit": UNIT, "us_per_step": e2e_s * 1e6,
                         "h2d_bytes_per_step": int(qh.numel() * qh.element_size()) + plan_bytes,
                         "d2h_bytes_per_step": int(oh.numel() * oh.element_size() + lh.numel() * 4),
                         "path": "psp_step_host: plan + plan upload + q H2D + run + o/lse D2H, synchronous; "
                                 "the K/V cache stays resident in HBM"}
        pipe_s, pipe_in, pipe_out = e2e_pipelined(psp, step, case, tens, ws, stream, args.steps, args.warmup)
        result["e2e_pipelined"] = {
            "value": world * ub / pipe_s / 1e9, "unit": UNIT, "us_per_step": pipe_s * 1e6,
            "h2d_bytes_per_step": pipe_in, "d2h_bytes_per_step": pipe_out,
            "path": "psp_plan + psp_upload + psp_run per step with q H2D and o/lse D2H through pinned host "
                    "buffers on copy streams; the host plans step i+1 while the device runs step i and "
                    "waits for step i's output one step later; no L2 flush (K/V larger than L2)"}
    step.close()
    del head, ws, tens

    # ---- the other workloads, measured in the same process (context for the headline line)
    if not args.no_per_config and rank == 0:
        per = {}
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            c = workloads.make_case(name, args.seed)
            r = measure_case(psp, runner, c, max(5, min(args.steps, 30)), 3)
            per[name] = config_summary(r, pk, pk_src)
            r["step"].close()
            del r
            torch.cuda.empty_cache()
        result["per_config"] = per

    # ---- CPU baseline: the oracle as it stands
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = oracle_timing(case, args.cpu_seconds)
        result["cpu_baseline"] = {"value": ub / ot["step_s"] / 1e9, "unit": UNIT, "cores": ot["cores"],
                                  "kind": "oracle", "us_per_step": ot["step_s"] * 1e6,
                                  "sample": f"{ot['rows']} of {ot['total_rows']} (request, head) rows"
                                            + (f", the whole step {ot['reps']} times" if ot["reps"] > 1 else "")
                                            + f", {ot['sample_s']:.1f} s of fp64 work on {ot['cores']} threads, "
                                            "scaled by context tokens"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))
    return 0


if __name__ == "__main__":
    sys.exit(main())
