#!/usr/bin/env python3
"""Throughput of the fused AdamW step with its gradient statistics on GB300.

One step is the whole hot path on the 1,073,741,824-parameter FP32 bucket with
BF16 gradients: row analysis (4,194,304 rows of 256), the fan-in-1024 merge,
the 12-byte report read back, the skip / global-norm clip decision
(max_grad_norm 1.0), and the fused update.  Inputs are synthetic and seeded,
resident in HBM before the timed region; each step moves ~30 GB, far more than
the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU: the ZeRO-1 data-parallel step over
an N x 1.07e9-parameter bucket (weak scaling: each rank owns a 1.07e9-parameter
shard of the optimizer state) -- a reduce-scatter of the ranks' gradients, the
shard's statistics, the 12-byte exchange and one global decision, the shard's
update, an all-gather of the parameters.  At N = 1 the bench checks its own
result: the oracle replays the timed run's sampled elements (the CPU leg) and a
failing check prints no value and exits non-zero.  ``--impl reference`` times
the CPU oracle on a bounded sample of the same workload (the pages publish no
implementation to run).  Prints one JSON line (rank 0).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused AdamW params/sec and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e datasheet bandwidth


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--next-rows-steps", type=int, default=10)
    # gloo stages the collectives through the host: for ranks sharing one GPU (testing)
    ap.add_argument("--dist-backend", choices=["nccl", "gloo"], default="nccl")
    # the ZeRO-1 step even on one rank (under torchrun: its collectives then stay on the GPU)
    ap.add_argument("--zero1", action="store_true")
    # (under torchrun spell it --params: torchrun's own parser takes --n for one of its flags)
    ap.add_argument("--params", "--n", dest="n", type=int, default=0,
                    help="override the parameter count (testing)")
    return ap.parse_args()


def workload(n_override=0):
    from synthetic.configs import CONFIG5
    w = CONFIG5
    if n_override:
        w = w.scaled(n_override)
    return w


def config_dict(w):
    return {"workload": w.name, "params": w.n, "param_dtype": "f32", "grad_dtype": w.grad_dtype,
            "optimizer": "adamw", "lr": w.lr, "betas": [w.beta1, w.beta2], "eps": w.eps,
            "weight_decay": w.weight_decay, "row_len": w.row_len, "merge_fan_in": 1024,
            "max_grad_norm": w.max_grad_norm, "gradient_scale": w.gradient_scale,
            "l2_policy": f"inputs larger than L2 (about {28 * w.n / 1e9:.0f} GB moved per step), "
                         "no flush"}


def update_kernel_traffic(n):
    """DRAM bytes per launch of the steady update kernel, from the committed ncu
    summary scaled to ``n`` parameters; None once the kernel source has changed
    since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "update_kernel_traffic_flat256M_bf16.txt")
    try:
        vals = {}
        for line in open(path):
            line = line.split("#", 1)[0].split()
            if len(line) == 2:
                vals[line[0]] = line[1]
        h = hashlib.sha256()
        for f in ("update_kernels.cu", "internal.h"):
            with open(os.path.join(ROOT, "amsgrad_optimizer_step_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        if h.hexdigest() != vals["source_sha256"]:
            return None
        per_param = (int(vals["dram_bytes_read"]) + int(vals["dram_bytes_write"])) / int(vals["params"])
        return per_param * n
    except Exception:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---- clocks during the timed region -------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd[1:1] = ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ---- CPU baseline: the oracle ---------------------------------------------------

def oracle_steps(w, sample: int, steps: int, warmup: int):
    """Times the oracle's whole step (global stats, decision, update) on ``sample``
    elements of the workload; returns (seconds per step, cores used)."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    idx = np.arange(sample)
    grads = [w.grad_host(c, idx) for c in (1, 2)]
    o = oracle.OracleAdamW(w.params_host(idx), w.options(), storage="f32", lib_=lib)
    times = []
    for k in range(warmup + steps):
        g = grads[k % 2]
        t0 = time.perf_counter()
        s, c = lib.gradient_stats(g, "bf16", w.gradient_scale)
        skip, _, coef = lib.clip_decision(s, c, w.max_grad_norm)
        o.step(g, "bf16", w.gradient_scale, skip_update=skip, clip_coef=coef)
        times.append(time.perf_counter() - t0)
    return statistics.median(times[warmup:]), 1


def host_info() -> dict:
    """CPU model, core count and architecture of the host."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"cpu": model or platform.processor() or "unknown", "cores": host_cores(),
            "machine": platform.machine()}


def gpu_info(dev) -> dict:
    import torch
    prop = torch.cuda.get_device_properties(dev)
    driver = None
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        driver = out.splitlines()[0] if out else None
    except Exception:
        pass
    return {"name": prop.name, "sms": prop.multi_processor_count,
            "memory_gib": round(prop.total_memory / 2 ** 30, 1), "driver": driver,
            "cuda_runtime": torch.version.cuda, "torch": torch.__version__}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_rank(conn, w, lo, hi):
    """One host core of the all-cores oracle run: it holds elements [lo, hi) of the
    workload and runs the oracle's step on them, statistics first, then the update
    with the decision the parent sends back."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    idx = np.arange(lo, hi)
    grads = [w.grad_host(c, idx) for c in (1, 2)]
    o = oracle.OracleAdamW(w.params_host(idx), w.options(), storage="f32", lib_=lib)
    conn.send("ready")
    while True:
        k = conn.recv()
        if k is None:
            break
        g = grads[k % 2]
        conn.send(lib.gradient_stats(g, "bf16", w.gradient_scale))
        skip, coef = conn.recv()
        o.step(g, "bf16", w.gradient_scale, skip_update=skip, clip_coef=coef)
        conn.send(True)
    conn.close()


def oracle_steps_all_cores(w, per_core: int, steps: int, warmup: int, cores: int):
    """The oracle on every host core, static contiguous chunks of ``per_core``
    elements, one process each (spawned: this may run after CUDA is initialised).
    A step is: every chunk's statistics, their sum and the decision in the parent,
    every chunk's update.  Returns seconds per step (median)."""
    import math
    import multiprocessing as mp
    import oracle
    lib = oracle.lib()
    ctx = mp.get_context("spawn")
    pipes, procs = [], []
    try:
        for r in range(cores):
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_oracle_rank, args=(b, w, r * per_core, (r + 1) * per_core),
                             daemon=True)
            pr.start()
            pipes.append(a)
            procs.append(pr)
        for a in pipes:
            if not a.poll(300):
                raise RuntimeError("an oracle worker did not start")
            a.recv()
        times = []
        for k in range(warmup + steps):
            t0 = time.perf_counter()
            for a in pipes:
                a.send(k)
            parts = [a.recv() for a in pipes]
            s = math.fsum(x[0] for x in parts)
            c = sum(int(x[1]) for x in parts)
            skip, _, coef = lib.clip_decision(s, c, w.max_grad_norm)
            for a in pipes:
                a.send((skip, coef))
            for a in pipes:
                a.recv()
            times.append(time.perf_counter() - t0)
        return statistics.median(times[warmup:])
    finally:
        for a in pipes:
            try:
                a.send(None)
            except Exception:
                pass
        for pr in procs:
            pr.join(timeout=10)
            if pr.is_alive():
                pr.kill()


def cpu_baseline(w, target_s=12.0):
    sample = 1 << 22
    sec, _ = oracle_steps(w, sample, steps=1, warmup=0)
    steps = max(2, int(0.4 * target_s / max(sec, 1e-3)))
    sec, _ = oracle_steps(w, sample, steps=steps, warmup=1)
    single = sample / sec
    cores = host_cores()
    per_core = 1 << 21
    out = {"value": single, "unit": UNIT, "cores": 1, "kind": "oracle",
           "single_core_value": single,
           "sample": f"{sample} elements of the {w.name} recipe (BF16 gradients, FP32 state), "
                     f"{steps} full steps (global stats + decision + update), single-threaded "
                     "FP64 C loop, median step"}
    if cores > 1:
        try:
            msteps = max(2, int(0.4 * target_s / max(sec * per_core / sample, 1e-3)))
            secm = oracle_steps_all_cores(w, per_core, msteps, 2, cores)
        except Exception as e:  # the single-core figure stands alone
            out["all_cores_error"] = str(e)[:200]
            return out
        out.update({"value": cores * per_core / secm, "cores": cores,
                    "sample": f"{cores} x {per_core} elements of the {w.name} recipe (BF16 "
                              f"gradients, FP32 state), one process per host core on a static "
                              f"chunk, {msteps} full steps (chunk statistics, summed decision, "
                              f"chunk updates), FP64 C loop, median step; single-threaded on "
                              f"{sample} elements: {single:.4g} params/s"})
    return out


def hbm_mix_rates(dev, n: int = 1 << 30, reps: int = 5) -> dict:
    """HBM rates (GB/s, best of ``reps``, CUDA events) of PyTorch's own streaming
    kernels, one per read:write byte mix, on buffers of n FP32 values (4 GiB each, far
    above L2): read only (sum), write only (fill), 1:1 (copy), 2:1 (add) and 1:2 (frexp:
    an FP32 value in, its FP32 mantissa and int32 exponent out).  HBM does not move every
    mix at the copy rate; these are the ceilings the fused kernels' own mixes are read
    against (the first step moves 6 B in and 12 B out per parameter, the analysis
    only reads)."""
    import torch
    a = torch.rand(n, device=dev)
    b = torch.rand(n, device=dev)
    c = torch.empty(n, device=dev)
    e = torch.empty(n, dtype=torch.int32, device=dev)
    ops = {"read_only": (lambda: a.sum(), 4), "write_only": (lambda: c.fill_(1.5), 4),
           "copy_1r_1w": (lambda: c.copy_(a), 8), "add_2r_1w": (lambda: torch.add(a, b, out=c), 12),
           "frexp_1r_2w": (lambda: torch.frexp(a, out=(c, e)), 12)}
    out = {}
    for name, (fn, bytes_per_elem) in ops.items():
        fn()
        best = float("inf")
        for _ in range(reps):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            fn()
            t1.record()
            torch.cuda.synchronize(dev)
            best = min(best, t0.elapsed_time(t1))
        out[name] = bytes_per_elem * n / (best * 1e-3) / 1e9
    del a, b, c, e
    torch.cuda.empty_cache()
    return out


def parity_indices(n: int, k: int = 40_000, seed: int = 0):
    """Sorted sample of element indices checked against the oracle: k seeded random
    ones plus both ends, the first vectors and 16-byte boundaries, the neighbours of
    the first edges of the full grid's 1024-element CTA stretches and of the pipeline's
    3072-element tiles, and the ragged end."""
    import numpy as np
    rng = np.random.default_rng(seed)
    base = set(rng.integers(0, n, k).tolist())
    for b in (0, 1, 2, 3, 4, 7, 8, 9, 1023, 1024, 1025, 2047, 2048, 2049,
              3071, 3072, 3073, 6143, 6144, 6145):
        base.add(b)
    for b in range(n - 9, n):
        base.add(b)
    return np.array(sorted(x for x in base if 0 <= x < n), dtype=np.int64)


def parity_check(w, snap, steps: int):
    """Replays the timed run's sampled elements through the oracle (the bench's CPU
    leg: with cpu_baseline, the only place the bench runs the oracle).

    ``snap`` holds, from the GPU run: the sampled indices, p, m, v there after
    ``steps`` statistics-guarded steps on the same gradient, the last report's norm
    and non-finite count, and a host copy of the whole gradient (produced by the
    seeded generator on the device; its sampled values are checked against the host
    generator first).  The oracle takes its own decision from its own FP64 sum over
    the whole gradient and runs ``steps`` updates on the sampled elements from the
    generator's initial parameters; the device must match within the trajectory
    tolerance |d| <= 1e-5 * max(1, |x|), the norm within relative 1e-5, the count and
    the skip decision exactly."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    idx = snap["idx"]
    gh = w.grad_host(1, idx)
    inputs_ok = bool(np.array_equal(snap["g_bits"][idx], gh))
    t0 = time.perf_counter()
    s_or, c_or = lib.gradient_stats(snap["g_bits"], "bf16", w.gradient_scale)
    skip_or, norm_or, coef_or = lib.clip_decision(s_or, c_or, w.max_grad_norm)
    stats_s = time.perf_counter() - t0
    o = oracle.OracleAdamW(w.params_host(idx), w.options(), storage="f32", lib_=lib)
    for _ in range(steps):
        o.step(gh, "bf16", w.gradient_scale, skip_update=skip_or, clip_coef=coef_or)
    errs = {}
    for name, dev, ref in (("p", snap["p"], o.p), ("m", snap["m"], o.state.m),
                           ("v", snap["v"], o.state.v)):
        ref = np.asarray(ref, np.float64)
        e = np.abs(np.asarray(dev, np.float64) - ref) / np.maximum(1.0, np.abs(ref))
        errs[name] = float(np.max(e)) if np.all(np.isfinite(e)) else float("inf")
    max_err = max(errs.values())
    norm_err = abs(snap["norm"] - norm_or) / norm_or if norm_or > 0 else abs(snap["norm"])
    ok = (inputs_ok and max_err <= 1e-5 and norm_err <= 1e-5 and snap["nonfinite"] == c_or
          and snap["skipped"] == skip_or and snap["t"] == (0 if skip_or else steps))
    return {"ok": bool(ok), "elements": int(len(idx)), "values_checked": int(3 * len(idx)),
            "steps": steps, "max_rel_err": max_err, "per_array": errs, "tolerance": 1e-5,
            "norm": snap["norm"], "norm_oracle": norm_or, "norm_rel_err": norm_err,
            "nonfinite": [snap["nonfinite"], c_or], "skip": [snap["skipped"], skip_or],
            "t": snap["t"], "inputs_match_generator": inputs_ok,
            "oracle_full_gradient_stats_s": stats_s,
            "what": "p, m, v at the sampled elements after the warm-up and timed steps vs the "
                    "oracle's own trajectory; its decision from its FP64 sum over every "
                    "gradient value.  Sampling is exact for the update: each element's update "
                    "depends only on its own values and the shared decision; the statistics "
                    "that couple the elements are checked over the whole gradient"}


def row_snapshot(idx, arrays, t):
    """Host copies of a row's state at the sampled elements (device side of the row
    checks); ``arrays`` maps a name to a device tensor or None."""
    import torch
    it = torch.as_tensor(idx, device=next(a for a in arrays.values() if a is not None).device)
    out = {k: (a[it].cpu().numpy() if a is not None else None) for k, a in arrays.items()}
    out["t"] = int(t)
    return out


def row_parity_check(rec):
    """Replays one timed next-row batch through the oracle (the bench's CPU leg).

    ``rec`` holds the row's workload recipe, the sampled indices, the device gradient
    at them, and the device state there before and after the batch (warm-up calls
    included).  The oracle starts from the state before, takes the batch's steps
    (t after - t before) with the same gradient, and must land on the state after
    within |d| <= 1e-5 * max(1, |x|); the sampled gradient must be the generator's.
    A per-segment clipped row also carries the segment table, the clip threshold and
    the whole gradient: each sampled element then takes its segment's coefficient
    from the oracle's own decision over that segment."""
    import numpy as np
    import oracle
    lib = oracle.lib()
    w, idx, b, a = rec["w"], rec["idx"], rec["before"], rec["after"]
    gh = w.grad_host(1, idx)
    inputs_ok = bool(np.array_equal(rec["g_bits"], gh))
    if rec.get("p0_from_generator"):
        inputs_ok = inputs_ok and bool(np.array_equal(b["p"], w.params_host(idx)))
    opts = w.options()
    steps = a["t"] - b["t"]
    # the elements' groups and their clip coefficients: one group without statistics,
    # else one per segment, with the oracle's own per-segment decision from its FP64
    # statistics over the segment's whole gradient
    groups, extra = [(np.arange(len(idx)), 1.0)], {}
    if rec.get("seg") is not None:
        seg = np.asarray(rec["seg"], np.int64)
        g_all = rec["g_full_bits"]
        inputs_ok = inputs_ok and bool(np.array_equal(g_all[idx], gh))
        decisions = [lib.clip_decision(*lib.gradient_stats(g_all[lo:hi], rec["gdt"],
                                                           w.gradient_scale),
                                       rec["max_grad_norm"])
                     for lo, hi in zip(seg[:-1], seg[1:])]
        inputs_ok = inputs_ok and not any(d[0] for d in decisions)  # none planted here
        kseg = np.searchsorted(seg, idx, side="right") - 1
        groups = [(np.flatnonzero(kseg == k), decisions[k][2]) for k in np.unique(kseg)]
        coefs = [d[2] for d in decisions]
        extra = {"segments": int(len(seg) - 1), "min_clip_coef_oracle": float(min(coefs))}
    refs = {"p": np.empty(len(idx)), "m": np.empty(len(idx)), "v": np.empty(len(idx))}
    if opts["amsgrad"]:
        refs["vmax"] = np.empty(len(idx))
    for sel, coef in groups:
        o = oracle.OracleAdamW(b["p"][sel], opts, storage="f32", lib_=lib)
        if b["t"] > 0:
            o.state = oracle.OracleState(t=b["t"], m=b["m"][sel], v=b["v"][sel],
                                         vmax=b["vmax"][sel] if opts["amsgrad"] else None)
        for _ in range(steps):
            o.step(gh[sel], rec["gdt"], w.gradient_scale, clip_coef=coef)
        refs["p"][sel], refs["m"][sel], refs["v"][sel] = o.p, o.state.m, o.state.v
        if opts["amsgrad"]:
            refs["vmax"][sel] = o.state.vmax
    errs = {}
    for name, ref in refs.items():
        e = np.abs(np.asarray(a[name], np.float64) - ref) / np.maximum(1.0, np.abs(ref))
        errs[name] = float(np.max(e)) if np.all(np.isfinite(e)) else float("inf")
    max_err = max(errs.values())
    ok = inputs_ok and steps > 0 and max_err <= 1e-5
    return {"ok": bool(ok), "elements": int(len(idx)), "steps": int(steps),
            "max_rel_err": max_err, "per_array": errs, "inputs_match_generator": inputs_ok,
            **extra}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload(args.n)
    cores = host_cores()
    if cores > 1:
        sample = cores * (1 << 21)
        sec = oracle_steps_all_cores(w, 1 << 21, args.steps, args.warmup, cores)
        what = (f"{cores} x {1 << 21} elements per step of the {w.name} recipe, one process "
                "per host core on a static chunk")
    else:
        sample = 1 << 22
        sec, cores = oracle_steps(w, sample, steps=args.steps, warmup=args.warmup)
        what = f"{sample} elements per step of the {w.name} recipe, single-threaded"
    value = sample / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": what},
            "host": host_info(),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- the GPU arm -----------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist
    import amsgrad_optimizer_step_gb300 as fa
    from amsgrad_optimizer_step_gb300 import build, sharded

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    distributed = world > 1 or (args.zero1 and "WORLD_SIZE" in os.environ)
    zero1 = world > 1 or args.zero1
    # one rank per GPU; ranks beyond the visible GPUs share them (testing with gloo)
    local = int(os.environ.get("LOCAL_RANK", "0")) % max(1, torch.cuda.device_count())
    if distributed:
        torch.cuda.set_device(local)
        if args.dist_backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    dev = torch.device("cuda", local)
    build.build()
    w = workload(args.n)
    n = w.n
    row_len = w.row_len
    opts = fa.options(**w.options())
    ctl = fa.control(w.gradient_scale)

    def max_over_ranks(x: float) -> float:
        # NCCL reduces device tensors, gloo host tensors
        tt = torch.tensor([x], dtype=torch.float64,
                          device=dev if args.dist_backend == "nccl" else "cpu")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())

    zstep = None
    if not zero1:
        # resident inputs: the whole bucket
        p = torch.empty(n, dtype=torch.float32, device=dev)
        w.fill_params_device(p)
        m = torch.empty_like(p)
        v = torch.empty_like(p)
        g = torch.empty(n, dtype=torch.bfloat16, device=dev)
        w.fill_grad_device(1, g)
    else:
        # ZeRO-1 data parallelism over a bucket of world x n parameters (weak scaling:
        # each rank owns an n-parameter shard of the optimizer state): replicated
        # parameters, each rank's own full gradient (its share of the batch: gradient
        # stream 1 + rank), reduce-scatter, shard statistics, the 12-byte exchange,
        # shard update, all-gather
        big = w.scaled(world * n)
        zstep = sharded.Zero1Step(world * n, opts, torch.bfloat16, dev, row_len=row_len,
                                  max_grad_norm=w.max_grad_norm,
                                  gradient_scale=w.gradient_scale)
        assert zstep.shard == n and zstep.padded == world * n
        p = torch.empty(zstep.padded, dtype=torch.float32, device=dev)
        big.fill_params_device(p)
        g = torch.empty(zstep.padded, dtype=torch.bfloat16, device=dev)
        big.fill_grad_device(1 + rank, g)
        m, v = zstep.m, zstep.v
    rows = fa.fa_stats_rows(n, row_len)
    rows_buf = fa.stats_buffer(rows, dev)
    scratch = fa.scratch_buffer(rows, dev)
    report = fa.stats_buffer(1, dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    state = {"t": 0}
    launches = {"n": 0}
    merge_kernels, _ = fa.fa_stats_plan(rows)

    rep_pinned = torch.empty((1, 3), dtype=torch.int32).pin_memory()
    rep_arrived = torch.cuda.Event()

    def step(ev=None):
        """analyse -> merge -> 12-byte report -> decision -> update.

        One GPU: the update is gated on the device by the same report, so it
        follows the merge without a host round trip; the host reads the report
        (pinned copy) meanwhile and advances t unless the step was skipped.
        Several ranks (or --zero1): the ZeRO-1 step (reduce-scatter, shard
        statistics, the exchange of the ranks' totals and one decision on the host,
        the shard's update, all-gather)."""
        if ev: ev[0].record(stream)
        if zstep is not None:
            d = zstep.step(p, g, events=ev[1:] if ev else None)
            launches["n"] += 1 + merge_kernels + (0 if d["skipped"] else 1)
            state["t"] = zstep.t
            state["last"] = (d["grad_norm"], d["nonfinite"], d["skipped"])
            return d["grad_norm"]
        fa.fa_analyze_gradient(g, row_len, rows_buf)
        fa.fa_merge_gradient_stats(rows_buf, rows, scratch, report)
        if ev: ev[1].record(stream)
        launches["n"] += 1 + merge_kernels
        rep_pinned.copy_(report, non_blocking=True)
        rep_arrived.record(stream)
        if ev: ev[2].record(stream)
        fa.fa_bucket_update(None, p, g, m, v, None, state["t"], opts, ctl, report=report,
                            max_grad_norm=w.max_grad_norm)
        launches["n"] += 1
        if ev: ev[3].record(stream)
        rep_arrived.synchronize()
        h = fa.FaStats.from_buffer_copy(rep_pinned.numpy().tobytes())
        skip, norm, _ = fa.fa_clip_decision(fa.fa_stats_sum_sq(h), int(h.nonfinite),
                                            w.gradient_scale, w.max_grad_norm)
        if not skip:
            state["t"] += 1
        state["last"] = (norm, int(h.nonfinite), bool(skip))
        return norm

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = None
    clocks = ClockSampler(gpu_uuid if rank == 0 else None)
    if rank == 0:
        clocks.start()
        time.sleep(0.5)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    launches["n"] = 0
    if distributed:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    end.record(stream)
    torch.cuda.synchronize(dev)
    wall_ms = (time.perf_counter() - wall0) * 1e3
    if distributed:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    clock_info = clocks.stop() if rank == 0 else None
    timed_launches = launches["n"]

    stats_ms = [e[0].elapsed_time(e[1]) for e in evs]
    update_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_each = [e[0].elapsed_time(e[3]) for e in evs]
    if distributed:
        total_ms = max_over_ranks(total_ms)

    # The timed run's state at sampled elements, for the oracle replay at the end
    # (parity_check); the gradient is the same in every step.
    parity_snap = None
    if world == 1:
        import numpy as np
        idx = parity_indices(n)
        it = torch.as_tensor(idx, device=dev)
        parity_snap = {"idx": idx, "p": p[it].cpu().numpy(), "m": m[it].cpu().numpy(),
                       "v": v[it].cpu().numpy(), "norm": state["last"][0],
                       "nonfinite": state["last"][1], "skipped": state["last"][2],
                       "t": state["t"], "steps": args.warmup + args.steps,
                       "g_bits": g.view(torch.int16).cpu().numpy().view(np.uint16)}

    # End to end through the public C-ABI call, the gradient coming from pinned
    # host memory every step.  Two device gradient buffers: the copy of step
    # k+1's gradient (side stream) overlaps step k's compute; every copy and
    # every 12-byte report read-back lies inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        # one pinned copy of n gradient elements; several ranks copy their full
        # (world x n) gradient as world copies of it, so the host holds 2 GiB per rank
        g_host = g[:n].cpu().pin_memory()
        g_dev = [g, torch.empty_like(g)]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        released = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]
        h2d_bytes = g.numel() * g.element_size()
        mailbox = fa.report_mailbox()

        def copy_in(dst):
            for c in range(world):
                dst[c * n:(c + 1) * n].copy_(g_host, non_blocking=True)

        def e2e_step(gb):
            if zstep is not None:
                zstep.step(p, gb)
                state["t"] = zstep.t
            else:
                state["t"], _ = fa.fa_bucket_step_clipped_gated(None, p, gb, m, v, None,
                                                                state["t"], opts, ctl,
                                                                w.max_grad_norm, row_len,
                                                                rows_buf, scratch, report,
                                                                mailbox)

        # the host-to-device link on its own (same buffer, same stream), for reading e2e
        ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_in(g_dev[1])
        ev_a.record(stream)
        copy_in(g_dev[1])
        ev_b.record(stream)
        torch.cuda.synchronize(dev)
        h2d_ms = ev_a.elapsed_time(ev_b)

        # per-step events on both streams (to tell a slowed copy from a slowed step)
        cp_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                 for _ in range(args.e2e_steps)]
        st_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                 for _ in range(args.e2e_steps)]

        def enqueue_copy_timed(b, k):
            with torch.cuda.stream(copy_stream):
                if used[b]:
                    copy_stream.wait_event(released[b])
                cp_ev[k][0].record(copy_stream)
                copy_in(g_dev[b])
                cp_ev[k][1].record(copy_stream)
                copied[b].record(copy_stream)

        def run_e2e(steps):
            host_step = []
            enqueue_copy_timed(0, 0)
            for k in range(steps):
                b = k % 2
                if k + 1 < steps:
                    enqueue_copy_timed((k + 1) % 2, k + 1)
                stream.wait_event(copied[b])
                st_ev[k][0].record(stream)
                h1 = time.perf_counter()
                e2e_step(g_dev[b])
                h2 = time.perf_counter()
                st_ev[k][1].record(stream)
                released[b].record(stream)
                used[b] = True
                host_step.append((h2 - h1) * 1e3)
            return host_step

        # untimed warm-up through the same call
        run_e2e(min(args.warmup, args.e2e_steps))
        torch.cuda.synchronize(dev)
        if distributed:
            dist.barrier()
        t0 = time.perf_counter()
        host_step = run_e2e(args.e2e_steps)
        torch.cuda.synchronize(dev)
        e2e_s = time.perf_counter() - t0
        copy_ms = statistics.median(e[0].elapsed_time(e[1]) for e in cp_ev)
        step_ms = statistics.median(e[0].elapsed_time(e[1]) for e in st_ev)
        if distributed:
            e2e_s = max_over_ranks(e2e_s)
        e2e = {"value": world * n * args.e2e_steps / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": 12,
               "ms_per_step": e2e_s * 1e3 / args.e2e_steps, "steps": args.e2e_steps,
               "h2d_copy_ms": h2d_ms, "h2d_gbs": h2d_bytes / (h2d_ms * 1e-3) / 1e9,
               "overlapped_copy_ms_median": copy_ms, "overlapped_step_ms_median": step_ms,
               "overlapped_copy_ms_max": max(e[0].elapsed_time(e[1]) for e in cp_ev),
               "host_step_ms_median": statistics.median(host_step),
               "host_step_ms_max": max(host_step),
               "warmup": min(args.warmup, args.e2e_steps),
               "what": ("pinned-host BF16 gradient copied in every step (side stream, double "
                        "buffered), then the C-ABI statistics-guarded step (analyse, merge, "
                        "12-byte report read back, update gated on the same decision); "
                        "wall clock") if zstep is None else
                       ("each rank's full pinned-host BF16 gradient copied in every step (side "
                        "stream, double buffered), then the ZeRO-1 step (reduce-scatter, shard "
                        "statistics, 12-byte exchange, shard update, all-gather); wall clock, "
                        "max over ranks")}

    # Next-row measurements on the same resident workload (update kernels only,
    # CUDA events per launch): the plain update and the fused low-precision
    # write-back (BF16 model copy, +2 B/param).
    next_rows = None
    row_checks = {}  # next rows replayed through the oracle in the CPU leg
    if args.next_rows_steps > 0 and not zero1:  # the single-GPU rows, at N = 1 only
        import numpy as np
        p_model = torch.empty(n, dtype=torch.bfloat16, device=dev)

        def timed(fn, k):
            for _ in range(2):
                fn()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
            torch.cuda.synchronize(dev)
            for i in range(k):
                ev[i].record(stream)
                fn()
            ev[k].record(stream)
            torch.cuda.synchronize(dev)
            return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(k))

        def plain():
            state["t"], _ = fa.fa_bucket_step(None, p, g, m, v, None, state["t"], opts, ctl, 1.0)

        def first():
            # t = 0: the first-step kernel (moments written, not read); t is not kept
            fa.fa_bucket_step(None, p, g, m, v, None, 0, opts, ctl, 1.0)

        def writeback():
            if fa.fa_bucket_update(None, p, g, m, v, None, state["t"], opts, ctl,
                                   p_model=p_model):
                state["t"] += 1

        peak, peak_kind = measured_peaks()
        rows_out = {}
        # the whole step as one C-ABI call (the form a user calls): the last merge posts
        # the report to a pinned mailbox and the update decides on the device, so no
        # stream operation sits between them
        one_call_mailbox = fa.report_mailbox()

        def one_call():
            state["t"], _ = fa.fa_bucket_step_clipped_gated(
                None, p, g, m, v, None, state["t"], opts, ctl, w.max_grad_norm, row_len,
                rows_buf, scratch, report, one_call_mailbox)

        ms = timed(one_call, args.next_rows_steps)
        sb = fa.bytes_per_param(2, False, False) * n + 2 * n + rows * 12 * 2
        rows_out["step_one_call_gated"] = {
            "ms": ms, "params_per_s": n / (ms * 1e-3), "bytes": sb,
            "achieved_gbs": sb / (ms * 1e-3) / 1e9, "frac": sb / (ms * 1e-3) / 1e9 / peak,
            "peak_kind": peak_kind,
            "what": "fa_bucket_step_clipped_gated: analysis, merges posting to the mailbox, "
                    "the update deciding on the device; CUDA events per call"}
        for name, fn, bpp_k in (("update_only", plain, fa.bytes_per_param(2, False, False)),
                                ("first_step", first, fa.bytes_per_param(2, False, True)),
                                ("f1_writeback_bf16", writeback,
                                 fa.bytes_per_param(2, False, False) + 2)):
            ms = timed(fn, args.next_rows_steps)
            gbs = bpp_k * n / (ms * 1e-3) / 1e9
            rows_out[name] = {"ms": ms, "bytes_per_param": bpp_k, "achieved_gbs": gbs,
                              "frac": gbs / peak, "peak_kind": peak_kind,
                              "params_per_s": n / (ms * 1e-3)}
        del p_model

        # the HBM ceiling of each read:write mix, measured with PyTorch's kernels: the
        # first step (6 B in, 12 B out per parameter) is read against the 1:2 mix
        mixes = hbm_mix_rates(dev)
        rows_out["hbm_mix_rates_gbs"] = mixes
        rows_out["first_step"]["frac_of_1r_2w_mix"] = (rows_out["first_step"]["achieved_gbs"]
                                                       / mixes["frexp_1r_2w"])

        # f2: the pages' staged baseline against the fused update, on FP32
        # gradients (the case their 48 -> 28 and 60 -> 36 B/param model is stated
        # for), AdamW and AMSGrad, same resident state.
        g32 = g.float()
        delta = torch.empty_like(p)
        vmax = torch.zeros_like(p)
        f2_bitwise = {}
        for ams in (False, True):
            o = fa.options(**dict(w.options(), amsgrad=ams))
            vm = vmax if ams else None

            def fused():
                state["t"], _ = fa.fa_adamw_step_inplace(p, g32, m, v, vm, state["t"], o, ctl)

            def staged():
                state["t"], _ = fa.fa_adamw_step_staged(p, g32, m, v, vm, state["t"], o, ctl,
                                                        delta)

            tag = "amsgrad" if ams else "adamw"
            fb = fa.bytes_per_param(4, ams, False)
            sb = 60 if ams else 48
            # A B B A: each variant timed before and after the other, averaged
            t_f1 = timed(fused, args.next_rows_steps)
            t_s1 = timed(staged, args.next_rows_steps)
            t_s2 = timed(staged, args.next_rows_steps)
            t_f2 = timed(fused, args.next_rows_steps)
            t_f, t_s = (t_f1 + t_f2) / 2, (t_s1 + t_s2) / 2
            # after the timed batches: one more step of each from the same state must
            # give the same bits (the staged kernels evaluate the fused FP32 operations)
            copies = [x.clone() for x in (p, m, v, vm) if x is not None]
            t_same = state["t"]
            fa.fa_adamw_step_inplace(p, g32, m, v, vm, t_same, o, ctl)
            fa.fa_adamw_step_staged(copies[0], g32, copies[1], copies[2],
                                    copies[3] if ams else None, t_same, o, ctl, delta)
            torch.cuda.synchronize(dev)
            same = all(torch.equal(a.view(torch.int32), b.view(torch.int32))
                       for a, b in zip([x for x in (p, m, v, vm) if x is not None], copies))
            state["t"] = t_same + 1
            f2_bitwise[tag] = bool(same)
            del copies
            rows_out[f"f2_staged_vs_fused_f32_{tag}"] = {
                "fused_ms": t_f, "staged_ms": t_s, "fused_bytes_per_param": fb,
                "staged_bytes_per_param": sb, "fused_gbs": fb * n / (t_f * 1e-3) / 1e9,
                "staged_gbs": sb * n / (t_s * 1e-3) / 1e9, "speedup": t_s / t_f,
                "byte_model_ratio": sb / fb, "kernels": {"fused": 1, "staged": 5 if ams else 4},
                "bitwise_equal_after_timing": f2_bitwise[tag]}
        del g32, delta, vmax

        # the 124,439,808-parameter in-place BF16 workload (AdamW, wd 0.01, 1 % of the
        # gradients x100): its own buffers, steady steps
        from synthetic.configs import CONFIG3
        n3 = CONFIG3.n
        p3 = torch.empty(n3, device=dev)
        CONFIG3.fill_params_device(p3)
        m3, v3 = torch.zeros_like(p3), torch.zeros_like(p3)
        g3 = torch.empty(n3, dtype=torch.bfloat16, device=dev)
        CONFIG3.fill_grad_device(1, g3)
        o3 = fa.options(**CONFIG3.options())
        s3 = {"t": 0}

        def inplace3():
            s3["t"], _ = fa.fa_adamw_step_inplace(p3, g3, m3, v3, None, s3["t"], o3, ctl)

        idx3 = parity_indices(n3, k=20_000, seed=3)
        arr3 = {"p": p3, "m": m3, "v": v3}
        before3 = row_snapshot(idx3, arr3, s3["t"])
        ms = timed(inplace3, args.next_rows_steps)
        row_checks["inplace_124M_bf16_adamw"] = {
            "w": CONFIG3, "idx": idx3, "gdt": "bf16", "p0_from_generator": True,
            "g_bits": g3[torch.as_tensor(idx3, device=dev)].view(torch.int16).cpu().numpy()
                        .view("uint16"),
            "before": before3, "after": row_snapshot(idx3, arr3, s3["t"])}
        b = fa.bytes_per_param(2, False, False)
        rows_out["inplace_124M_bf16_adamw"] = {
            "ms": ms, "params": n3, "bytes_per_param": b,
            "achieved_gbs": b * n3 / (ms * 1e-3) / 1e9,
            "frac": b * n3 / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "params_per_s": n3 / (ms * 1e-3)}
        del p3, m3, v3, g3

        # f4: the torch.optim-style wrapper on the decoder-shaped 1.196e9-parameter
        # model (199 FP32 tensors packed into one bucket), global clip 1.0: each
        # step analyses, merges, reads back 12 bytes, decides and updates.
        from amsgrad_optimizer_step_gb300.optim import FusedAdamW
        from synthetic.configs import decoder_bucket_shapes
        dparams = [torch.nn.Parameter(torch.zeros(shape, device=dev))
                   for _, shape in decoder_bucket_shapes()]
        dn = sum(x.numel() for x in dparams)
        dopt = FusedAdamW(dparams, lr=1e-3, max_grad_norm=1.0)
        dopt._buckets[0].grad.normal_(0.0, 1e-3)
        ms = timed(dopt.step, args.next_rows_steps)
        b4 = fa.bytes_per_param(4, False, False) + 4  # update + analysis read of the FP32 gradient
        rows_out["f4_fused_adamw_decoder1.1B_clip"] = {
            "ms": ms, "params": dn, "tensors": len(dparams), "row_len": dopt.row_len,
            "bytes_per_param": b4, "achieved_gbs": b4 * dn / (ms * 1e-3) / 1e9,
            "frac": b4 * dn / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "params_per_s": dn / (ms * 1e-3), "skipped": dopt.last_report["skipped"]}
        del dopt, dparams
        torch.cuda.empty_cache()

        # the same model in mixed precision: BF16 parameters and gradients, FP32 masters
        # and moments, the BF16 copy written back in the update's pass
        dparams = [torch.nn.Parameter(torch.zeros(shape, device=dev, dtype=torch.bfloat16))
                   for _, shape in decoder_bucket_shapes()]
        dopt = FusedAdamW(dparams, lr=1e-3, max_grad_norm=1.0)
        dopt._buckets[0].grad.normal_(0.0, 1e-3)
        ms = timed(dopt.step, args.next_rows_steps)
        b4 = fa.bytes_per_param(2, False, False) + 2 + 2  # update + model copy + analysis
        rows_out["f4_fused_adamw_decoder1.1B_bf16_params_clip"] = {
            "ms": ms, "params": dn, "tensors": len(dparams), "row_len": dopt.row_len,
            "bytes_per_param": b4, "achieved_gbs": b4 * dn / (ms * 1e-3) / 1e9,
            "frac": b4 * dn / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "params_per_s": dn / (ms * 1e-3), "skipped": dopt.last_report["skipped"]}
        del dopt, dparams
        torch.cuda.empty_cache()

        # f3: per-parameter clipping on the decoder-shaped bucket (199 segments,
        # FP16 gradients, AMSGrad): segment-aligned analysis, one report per
        # segment, 199 x 12 bytes read back, per-segment clip, update.
        from synthetic.configs import CONFIG4, decoder_bucket_offsets
        seg = [int(x) for x in decoder_bucket_offsets()]
        sn = seg[-1]
        sp = torch.empty(sn, device=dev)
        CONFIG4.fill_params_device(sp)
        sm, sv, svm = (torch.zeros(sn, device=dev) for _ in range(3))
        sg = torch.empty(sn, dtype=torch.float16, device=dev)
        CONFIG4.fill_grad_device(1, sg)
        crow = fa.segment_rows(seg, 512)
        srows = fa.stats_buffer(crow[-1], dev)
        sscr = torch.empty(fa.fa_stats_chunk_scratch(crow), device=dev)
        srep = fa.stats_buffer(len(seg) - 1, dev)
        so = fa.options(**CONFIG4.options())
        sstate = {"t": 0, "rep": None}

        def per_segment_host():
            sstate["t"], sstate["rep"], _, _ = fa.fa_bucket_step_clipped_per_segment(
                seg, sp, sg, sm, sv, svm, sstate["t"], so, ctl, 0.01, 512, srows, sscr, srep)

        # the same step decided on the device: the 199 reports are copied to pinned
        # memory right behind the merges; every segment's decision is then taken once in
        # the merge scratch (free again) and the update runs on the full grid reading
        # it, without waiting for the host, which reads the reports only to advance the
        # step count
        srep_pinned = torch.empty(srep.shape, dtype=srep.dtype).pin_memory()
        srep_ready = torch.cuda.Event()

        def per_segment():
            fa.fa_analyze_gradient(sg, 512, srows, seg)
            fa.fa_merge_gradient_stats_chunks(srows, crow, sscr, srep)
            srep_pinned.copy_(srep, non_blocking=True)
            srep_ready.record(stream)
            fa.fa_bucket_update(seg, sp, sg, sm, sv, svm, sstate["t"], so, ctl, seg_reports=srep,
                                max_grad_norm=0.01, seg_decided=sscr)
            srep_ready.synchronize()
            if not bool((srep_pinned[:, 1] != 0).any()):
                sstate["t"] += 1

        from synthetic.configs import CONFIG4_MAX
        edges4 = sorted({x + d for x in seg[1:-1] for d in (-1, 0)})
        idx4 = np.unique(np.concatenate([parity_indices(sn, k=20_000, seed=4),
                                         np.asarray(edges4, np.int64)]))
        g4_bits = sg[torch.as_tensor(idx4, device=dev)].view(torch.int16).cpu().numpy().view("uint16")
        g4_all = sg.view(torch.int16).cpu().numpy().view("uint16")  # the oracle's statistics
        arr4 = {"p": sp, "m": sm, "v": sv, "vmax": svm}
        seg_clip = {"seg": seg, "max_grad_norm": 0.01, "g_full_bits": g4_all}
        before_f3 = row_snapshot(idx4, arr4, sstate["t"])
        # and as one call, the host reading the bucket's record from a mailbox that the
        # decision kernel posts before the update runs
        f3_mailbox = fa.report_mailbox()

        def per_segment_one_call():
            fa.fa_bucket_step_clipped_per_segment_gated(seg, sp, sg, sm, sv, svm, sstate["t"],
                                                        so, ctl, 0.01, 512, srows, sscr, srep,
                                                        mailbox=f3_mailbox)
            if int(f3_mailbox[1]) == 0:  # the bucket's non-finite count
                sstate["t"] += 1

        ms_host = timed(per_segment_host, args.next_rows_steps)
        min_coef = sstate["rep"].clip_coef
        after_f3_host = row_snapshot(idx4, arr4, sstate["t"])
        ms = timed(per_segment, args.next_rows_steps)
        ms_one_call = timed(per_segment_one_call, args.next_rows_steps)
        row_checks["f3_per_segment_clip_decoder1.1B_f16_amsgrad/host_decided"] = dict(
            seg_clip, w=CONFIG4, idx=idx4, gdt="f16", g_bits=g4_bits, p0_from_generator=True,
            before=before_f3, after=after_f3_host)
        row_checks["f3_per_segment_clip_decoder1.1B_f16_amsgrad"] = dict(
            seg_clip, w=CONFIG4, idx=idx4, gdt="f16", g_bits=g4_bits, before=after_f3_host,
            after=row_snapshot(idx4, arr4, sstate["t"]))
        b3 = fa.bytes_per_param(2, True, False) + 2  # AMSGrad update + analysis read of the FP16 gradient
        rows_out["f3_per_segment_clip_decoder1.1B_f16_amsgrad"] = {
            "ms": ms, "params": sn, "segments": len(seg) - 1, "row_len": 512,
            "bytes_per_param": b3, "achieved_gbs": b3 * sn / (ms * 1e-3) / 1e9,
            "frac": b3 * sn / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
            "params_per_s": sn / (ms * 1e-3), "min_clip_coef": min_coef,
            "decided": "on the device, once per segment", "host_decided_ms": ms_host,
            "one_call_ms": ms_one_call}
        # the same bucket without statistics (AMSGrad, FP16 gradients, one launch over
        # 199 tensors), maximize off and on
        for tag, cfg in (("", CONFIG4), ("_maximize", CONFIG4_MAX)):
            ob = fa.options(**cfg.options())

            def bucket():
                sstate["t"], _ = fa.fa_bucket_step(seg, sp, sg, sm, sv, svm, sstate["t"], ob,
                                                   ctl, 1.0)

            before4 = row_snapshot(idx4, arr4, sstate["t"])
            ms = timed(bucket, args.next_rows_steps)
            row_checks["bucket_decoder1.1B_f16_amsgrad" + tag] = {
                "w": cfg, "idx": idx4, "gdt": "f16", "g_bits": g4_bits,
                "before": before4, "after": row_snapshot(idx4, arr4, sstate["t"])}
            b = fa.bytes_per_param(2, True, False)
            rows_out["bucket_decoder1.1B_f16_amsgrad" + tag] = {
                "ms": ms, "params": sn, "tensors": len(seg) - 1, "bytes_per_param": b,
                "achieved_gbs": b * sn / (ms * 1e-3) / 1e9,
                "frac": b * sn / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
                "params_per_s": sn / (ms * 1e-3)}
        del sp, sm, sv, svm, sg, srows, sscr, srep
        torch.cuda.empty_cache()
        next_rows = rows_out

    if rank == 0:
        ms_step = total_ms / args.steps
        bpp = fa.bytes_per_param(2, False, False)
        upd_ms = statistics.median(update_ms)
        st_ms = statistics.median(stats_ms)
        peak, peak_kind = measured_peaks()
        achieved = bpp * n / (upd_ms * 1e-3) / 1e9
        step_bytes = bpp * n + 2 * n + rows * 12 * 2
        line = {
            "metric": METRIC, "value": world * n / (ms_step * 1e-3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(w),
            "achieved_gbs_step": step_bytes / (ms_step * 1e-3) / 1e9,
            "roofline": {"bound": "hbm",
                         "kernel": "update_vec_cta_gate_kernel (fused AdamW, BF16 grad, steady state, "
                                   "gated on the device report; full grid of 64-thread CTAs)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                         "target": ">= 0.80 of the nominal ~8 TB/s HBM3e peak, i.e. frac_of_nominal; "
                                   "frac is against the measured copy peak",
                         "bytes_per_param": bpp, "traffic": update_kernel_traffic(n),
                         "kernel_ms_median": upd_ms, "kernel_ms_min": min(update_ms),
                         "kernel_ms_max": max(update_ms)},
            "step_ms": {"median": statistics.median(step_each), "min": min(step_each),
                        "max": max(step_each), "samples": len(step_each)},
            "wall_clock": {"ms_per_step": wall_ms / args.steps,
                           "what": "host clock over the timed steps: submission, the "
                                   "12-byte read-back and the decision included"},
            "stats_path": {"ms_median": st_ms, "analyze_bytes": n * 2 + rows * 12,
                           "achieved_gbs": (n * 2 + rows * 12) / (st_ms * 1e-3) / 1e9,
                           "what": "analysis and merges, CUDA events inside the step (with "
                                   "the reduce-scatter at N > 1); a read-only stream, read "
                                   "against next_rows.hbm_mix_rates_gbs.read_only"},
            "gpu_launches": timed_launches,
            "clocks": clock_info,
            "host": host_info(),
            "gpu": gpu_info(dev),
            "e2e": e2e,
            "next_rows": next_rows,
        }
        if zero1:
            line["config"]["parallelism"] = f"dp{world}, ZeRO-1 (optimizer state sharded)"
        if world > 1:
            line["parity"] = {"ok": None, "checked": False,
                              "why": "the oracle runs in the CPU leg at N = 1 only; the "
                                     "ZeRO-1 step is checked against the oracle over the whole "
                                     "bucket by the logical-rank tests"}
        rc = 0
        if parity_snap is not None:  # the CPU leg: the oracle replays the sampled elements
            par = parity_check(w, parity_snap, parity_snap["steps"])
            if next_rows is not None:
                par["f2_staged_equals_fused_bitwise"] = f2_bitwise
                par["ok"] = par["ok"] and all(f2_bitwise.values())
                rows_par = {name: row_parity_check(rec) for name, rec in row_checks.items()}
                for name, rp in rows_par.items():
                    row, _, variant = name.partition("/")
                    next_rows[row]["parity_" + variant if variant else "parity"] = rp
                par["next_rows_ok"] = {name: rp["ok"] for name, rp in rows_par.items()}
                par["ok"] = par["ok"] and all(rp["ok"] for rp in rows_par.values())
            line["parity"] = par
            if not par["ok"]:  # an unchecked or failing number is never reported
                line["value"] = None
                line["e2e"] = None
                rc = 1
        if not args.no_cpu_baseline and world == 1 and rc == 0:  # rank 0 at N = 1 only
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
        if rc:
            return rc
    if distributed:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
