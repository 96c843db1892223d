#!/usr/bin/env python3
"""Benchmark of one paged shared-prefix decode-attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--page-size P]
                    [--impl reference]

A step is one call of psp_run over the whole synthetic batch: the prefix
kernel of the shared-prefix group (dense or cascade branch, chosen by the
dispatcher) and the split-KV suffix kernel, whose last arriving CTA per
(request, KV head) performs the log-sum-exp merge, with the K/V pool, the
queries and the uploaded plan resident in HBM.  The metric is device time per
step and the achieved HBM bandwidth on the step's unique K/V bytes (a shared
prefix page counts once).  L2 is flushed (a buffer of twice the L2 size is
written and read back) between timed steps, outside the timed events.  The
default workload is the Llama-3.1-8B-shaped layer without sharing (B=32,
32/8 heads, bf16, contexts U[2048,4096], page size 16); --workload selects
the shared-prefix batches.

Printed (rank 0, one JSON line): value = unique-KV GB/s over all ranks,
us_per_step, the dominant kernel's roofline, the oracle's CPU baseline, the
end-to-end figure through psp_step_host with host buffers (plan, plan upload,
query copy in, output copy out, every step), sampled SM clocks, the launch
count, a bare read of the same byte count for context (read_ceiling), and for
shared-prefix workloads the per-request paged comparator (every request
reading the prefix through its own block table).

--impl reference times the fp64 CPU oracle (the reference arm of this path)
on a bounded sample of the same workload, in the same metric and unit.
Multi-GPU (torchrun): independent replicas, one per GPU, no collective in the
step; value = units of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
KERNEL_SOURCES = {
    "suffix_splitkv": "paged_shared_prefix_gb300/csrc/kernel_suffix.cu",
    "prefix_cascade": "paged_shared_prefix_gb300/csrc/kernel_prefix_cascade.cu",
    "prefix_dense": "paged_shared_prefix_gb300/csrc/kernel_prefix_dense.cu",
    "expand_kv_indices": "paged_shared_prefix_gb300/csrc/kernel_merge.cu",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama8b_noshare", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--page-size", type=int, default=None)
    ap.add_argument("--impl", default="psp", choices=["psp", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--threshold", type=int, default=0, help="dense/cascade M_eff threshold (0 = built-in)")
    ap.add_argument("--token-flat", action="store_true", help="lower to per-token kv_indices inside the step")
    ap.add_argument("--concurrent", type=int, default=None,
                    help="1: prefix kernels on a side stream concurrent with the suffix kernel, 0: one stream "
                         "(default: the library default for the workload)")
    ap.add_argument("--no-comparator", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-ceiling", action="store_true", help="skip the bare-read ceiling measurement")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target oracle CPU time for the baseline")
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


def src_hash(rel: str) -> str:
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return ""


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(f"{kernel}@{workload}")
    if not ent or ent.get("source_sha256_16") != src_hash(KERNEL_SOURCES.get(kernel, "")):
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
    case = workloads.make_case(args.workload, args.seed, page_size=args.page_size)
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
    """Dispatcher refit: for a 4096-token prefix and 8 KV heads, time the prefix kernel of
    both branches over batch x GQA group; the threshold is the smallest swept M_eff from
    which the dense branch is never slower than the cascade branch."""
    import torch

    import paged_shared_prefix_gb300 as psp
    dev = torch.device("cuda:0")
    rows = []
    for G in (1, 2, 4, 8):
        for B in (4, 8, 16, 32, 64, 128, 256, 512):
            m_eff = B * G
            if m_eff < 16 or m_eff > 4096:
                continue
            case = workloads.make_case("agent", 11, batch=B, prefix_len=4096, private_range=(1, 16),
                                       num_q_heads=8 * G, num_kv_heads=8)
            tens = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev))
                    for k, v in dict(q=case.q, k=case.k_pool, v=case.v_pool).items()}
            o = torch.empty((B, 8 * G, 128), dtype=torch.bfloat16, device=dev)
            res = {}
            for branch, thr in (("dense", 1), ("cascade", 1 << 30)):
                step = psp.DecodeStep.for_case(case, dense_threshold=thr)
                step.plan_case(case)
                ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
                step.upload(ws)
                step.set_kernel_timing(True)
                times = []
                for i in range(8):
                    step.run(tens["q"], tens["k"], tens["v"], o)
                    torch.cuda.synchronize()
                    if i >= 3:
                        times += [ms for n, ms in step.kernel_times() if n.startswith("prefix")]
                res[branch] = statistics.median(times) * 1e3
                step.close()
            rows.append({"G": G, "B": B, "m_eff": m_eff, "dense_us": res["dense"], "cascade_us": res["cascade"]})
    rows.sort(key=lambda r: r["m_eff"])
    thr = None
    for i, r in enumerate(rows):
        if all(x["dense_us"] <= x["cascade_us"] for x in rows[i:]):
            thr = r["m_eff"]
            break
    print(json.dumps({"sweep": rows, "refit_threshold": thr,
                      "gpu": torch.cuda.get_device_name(0), "prefix_tokens": 4096, "kv_heads": 8}))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep_threshold:
        return sweep_threshold(args)

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

    case = workloads.make_case(args.workload, args.seed + rank, page_size=args.page_size)
    w = case.workload
    ub = workloads.unique_kv_bytes(case)
    paged_b = workloads.paged_kv_bytes(case)

    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    q, kp, vp, ks, vs = t(case.q), t(case.k_pool), t(case.v_pool), t(case.k_scale), t(case.v_scale)
    odt = torch.float32 if w.o_dtype == "f32" else torch.bfloat16
    o = torch.empty((case.batch, w.num_q_heads, w.head_dim), dtype=odt, device=dev)
    lse = torch.empty((case.batch, w.num_q_heads), dtype=torch.float32, device=dev)

    concurrent = bool(args.concurrent) if args.concurrent is not None else False
    step = psp.DecodeStep.for_case(case, dense_threshold=args.threshold, token_flat=args.token_flat,
                                   concurrent=concurrent)
    t_plan = []
    for _ in range(5):
        t0 = time.perf_counter()
        step.plan_case(case)
        t_plan.append(time.perf_counter() - t0)
    info = step.plan_info()
    ws = torch.empty(step.workspace_size(), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    step.upload(ws, stream)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer of twice the L2 size (evicts the step's data), then read it back so
        # no dirty line is left whose write-back would land inside the next timed step
        flush.fill_(1.0)
        torch.sum(flush, dim=0, out=sink)

    def one(timed_events=None):
        flush_l2()
        if timed_events:
            timed_events[0].record(stream)
        step.run(q, kp, vp, o, lse, ks, vs, stream)
        if timed_events:
            timed_events[1].record(stream)

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()

    # ---- timed region: whole steps, no per-kernel events (they would sit between the prefix
    # and suffix kernels and stop the suffix kernel from starting early)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        one(evs[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms, value = aggregate_replicas(statistics.mean(step_ms), ub, world, dev)

    # ---- per-kernel times (events on the launching stream around each kernel), a separate pass
    step.set_kernel_timing(True)
    kern = {}
    n_kernel_steps = max(3, min(args.steps, 20))
    for i in range(n_kernel_steps):
        one()
        torch.cuda.synchronize()
        for name, kms in step.kernel_times():
            kern.setdefault(name, []).append(kms)
    step.set_kernel_timing(False)
    launches = args.steps * sum(len(v) for v in kern.values()) // n_kernel_steps

    # ---- single-launch read ceiling: a bare read of as many bytes as the step's unique K/V
    # (torch's sum kernel, L2 flushed the same way), for context beside the roofline peak
    ceil = None
    if not args.no_read_ceiling:
        buf = torch.empty(ub // 4, dtype=torch.float32, device=dev).fill_(1.0)
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(8)]
        for i in range(10):
            flush_l2()
            if i >= 2:
                cev[i - 2][0].record(stream)
            torch.sum(buf, dim=0, out=sink)
            if i >= 2:
                cev[i - 2][1].record(stream)
        torch.cuda.synchronize()
        cms = statistics.mean(a.elapsed_time(b) for a, b in cev)
        ceil = {"gbs": buf.numel() * 4 / (cms * 1e-3) / 1e9, "bytes": int(buf.numel() * 4),
                "how": "torch.sum over a float32 buffer of the unique K/V size, one launch, L2 flushed as for the step"}
        del buf

    # ---- roofline of the dominant kernel
    pk, pk_src = peaks()
    kmean = {k: statistics.mean(v) for k, v in kern.items()}
    dom = max(kmean, key=kmean.get)
    Hkv, d = w.num_kv_heads, w.head_dim
    elem = workloads.elem_bytes(w.kv_dtype)
    tok_bytes = 2 * Hkv * d * elem
    if dom in ("prefix_dense", "prefix_cascade"):
        m_eff = int(case.batch * (w.num_q_heads // Hkv))
        flops = 4.0 * m_eff * info["shared_tokens"] * d * Hkv
        achieved = flops / (kmean[dom] * 1e-3) / 1e12
        peak = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        peak_note = pk_src
        if w.kv_dtype == "fp8_e4m3" and dom == "prefix_dense":
            # e4m3 products: the measured bf16 peak times the nominal fp8 / bf16 ratio (4.5 / 2.25)
            peak *= 2.0
            peak_note = f"{pk_src} bf16 x 2 (nominal e4m3 / bf16 ratio)"
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic(dom, w.name), "kernel": dom,
                "algorithmic": f"{flops:.4g} FLOP per launch (4*M_eff*P*d*Hkv)", "peak_source": peak_note}
    else:
        if dom == "suffix_splitkv":
            alg = info["suffix_tokens"] * tok_bytes
            desc = f"{alg} B per launch = {info['suffix_tokens']} suffix tokens x {tok_bytes} B (K+V, all KV heads)"
        else:
            alg = ub
            desc = f"{alg} unique K/V bytes"
        achieved = alg / (kmean[dom] * 1e-3) / 1e9
        peak = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(dom, w.name), "kernel": dom, "algorithmic": desc,
                "peak_source": pk_src}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "f32", "bf16": "bf16", "fp8_e4m3": "fp8_e4m3"}[w.kv_dtype],
        "data": "synthetic",
        "config": {"workload": describe(case), "l2": "flushed between steps (2x L2 buffer written then read back, untimed)",
                   "parallelism": f"replicas x{world}", "token_flat": bool(args.token_flat),
                   "concurrent_prefix": concurrent},
        "unique_kv_bytes": ub, "paged_kv_bytes": paged_b,
        "hbm_frac_of_8tbs": value / world / 8000.0,
        "kernels_ms": kmean, "plan_us": statistics.median(t_plan) * 1e6,
        "roofline": roof, "read_ceiling": ceil, "clocks": clk, "gpu_launches": launches, "wall_s": wall,
        "plan": {k: info[k] for k in ("num_splits", "num_chunks", "suffix_ctas", "prefix_dense_ctas",
                                       "prefix_cascade_ctas", "dense_threshold", "num_sms")},
    }

    # ---- per-request paged comparator (prefix read through every block table)
    if not args.no_comparator and case.num_groups > 0:
        nc = case.without_sharing()
        cstep = psp.DecodeStep.for_case(nc, token_flat=args.token_flat)
        cstep.plan_case(nc)
        cws = torch.empty(cstep.workspace_size(), dtype=torch.uint8, device=dev)
        cstep.upload(cws, stream)
        ce = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
        for i in range(13):
            flush_l2()
            if i >= 3:
                ce[i - 3][0].record(stream)
            cstep.run(q, kp, vp, o, lse, ks, vs, stream)
            if i >= 3:
                ce[i - 3][1].record(stream)
        torch.cuda.synchronize()
        cms = statistics.mean(a.elapsed_time(b) for a, b in ce)
        result["paged_comparator"] = {"us_per_step": cms * 1e3, "speedup_read_once": cms / ms,
                                      "bytes_per_step": paged_b}
        cstep.close()

    # ---- end to end through the C ABI with host buffers
    if not args.no_e2e:
        qh = torch.from_numpy(np.ascontiguousarray(case.q).view(np.int16 if w.q_dtype == "bf16" else np.float32))
        qh = qh.pin_memory()
        oh = torch.empty(o.shape, dtype=torch.int16 if w.o_dtype == "bf16" else torch.float32).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        qd = torch.empty_like(q)
        batch, keep = step.make_batch(case.kv_len, case.page_indptr, case.page_indices, case.prefix_group,
                                      case.group_prefix_len)
        devt = step.tensors(qd, kp, vp, o, lse, ks, vs)
        e2e = []
        for i in range(3 + args.steps):
            flush_l2()
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

    # ---- CPU baseline: the oracle as it stands
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = oracle_timing(case, args.cpu_seconds)
        result["cpu_baseline"] = {"value": ub / ot["step_s"] / 1e9, "unit": UNIT, "cores": ot["cores"],
                                  "kind": "oracle", "us_per_step": ot["step_s"] * 1e6,
                                  "sample": f"{ot['rows']} of {ot['total_rows']} (request, head) rows"
                                            + (f", the whole step {ot['reps']} times" if ot["reps"] > 1 else "")
                                            + f", {ot['sample_s']:.1f} s of fp64 work on {ot['cores']} threads, "
                                            "scaled by context tokens"}
    step.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))
    return 0


if __name__ == "__main__":
    sys.exit(main())
