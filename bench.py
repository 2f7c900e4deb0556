#!/usr/bin/env python
"""Benchmark of the Ozaki Scheme II emulated DGEMM on GB300.

Metric: emulated-DGEMM TFLOP/s = 2 m n k / t for C = A B with m = n = k = 8192,
entries (U(0,1) - 0.5) exp(0.5 N(0,1)) (seed = rank), 16 moduli, revised fast
mode.  One step = one os2_gemm call (all five steps of the method) with the
inputs already resident in HBM; `e2e` is the same metric through
os2_gemm_host with the inputs and the result in pinned host memory (copies
inside the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun: every rank multiplies its own independent pair of
matrices (no collective on the data path; weak scaling), timing is bracketed
by barriers and the max over ranks is reported.

The line also carries `int8_tensor_path`: the same product with step 3 on
the INT8 tensor path (mma.sync s8), its rate against the mma.sync s8 probe.

`--impl reference` times the CPU oracle (the exact reference implementation of
the method) on the host cores, on a bounded sample of output entries of the
same workload; only rank 0 runs it.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "emulated-DGEMM TFLOP/s (2mnk/t) at 8192^3 & INT8 tensor-pipe utilisation"
UNIT = "TFLOP/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--m", type=int, default=8192)
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--k", type=int, default=8192)
    ap.add_argument("--num-moduli", type=int, default=16)
    ap.add_argument("--mode", default="fast", choices=["fast", "accurate"])
    ap.add_argument("--phi", type=float, default=0.5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip native DGEMM / accuracy context")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the N in {14,16,18} x {fast, accurate} sweep of the same workload")
    ap.add_argument("--e2e-calls", type=int, default=150,
                    help="timed os2_gemm_host calls of the e2e measurement (about 12 ms each at "
                         "8192^3; every call counts, stalls included)")
    ap.add_argument("--no-int8", action="store_true",
                    help="skip the short run of step 3 on the INT8 tensor path (mma.sync s8) "
                         "that gives the metric's INT8 tensor-pipe utilisation")
    ap.add_argument("--no-peaks", action="store_true",
                    help="skip the tensor-pipe peak probes (own kernels) before the timed steps")
    ap.add_argument("--crt", default="default", choices=["default", "tc", "simt", "auto"],
                    help="kernel of steps 4 + 5 (os2_set_crt_variant); default: the library's")
    ap.add_argument("--gemm", default="tc", choices=["tc", "tc_1sm", "tc_i8", "s8", "simt"],
                    help="step-3 kernel (os2_set_gemm_variant): tc (default), tc_1sm, tc_i8 "
                         "(int8 residue planes widened on chip), s8 (mma.sync s8 on int8 "
                         "planes; its roofline is the own mma.sync s8 probe) or simt")
    ap.add_argument("--accuracy", action="store_true",
                    help="error against the exact product for 1024^3, phi in {0.5,2,4}, N in "
                         "{12..20}, both modes, beside native DGEMM; prints one JSON line")
    ap.add_argument("--peaks-only", action="store_true",
                    help="run only the tensor-pipe peak probes and print them as one JSON line")
    return ap.parse_args()


def workload_name(a):
    return (f"{a.m}x{a.n}x{a.k} FP64 GEMM, entries (U(0,1)-0.5)*exp({a.phi}*N(0,1)), "
            f"{a.num_moduli} moduli, {a.mode} mode")


def config(a, extra=None):
    c = {"workload": workload_name(a), "m": a.m, "n": a.n, "k": a.k, "num_moduli": a.num_moduli,
         "mode": a.mode, "phi": a.phi, "seed": "rank",
         "l2": ("inputs larger than L2 (A and B %d MiB each), no flush" % (a.m * a.k * 8 >> 20))
         if a.m * a.k * 8 > 129e6 else "inputs smaller than L2 (no flush): small-case run"}
    if extra:
        c.update(extra)
    return c


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", uuid], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# -------------------------------------------------------------- utilities --
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_traffic(kernel: str, workload_key: str):
    """DRAM bytes per launch from a committed ncu capture, if it is for this
    workload and the sources that decide the kernel and its launches are
    unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh).get(kernel)
    if not d or d.get("workload_key") != workload_key:
        return None
    if not isinstance(d.get("sources_sha256"), dict) or "bytes_per_launch" not in d:
        return None
    for rel, want in d["sources_sha256"].items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest() != want:
            return None
    return d["bytes_per_launch"]


def exact_dot(a, b):
    """Correctly rounded sum_h a_h b_h (Dekker products + math.fsum)."""
    p = a * b
    c = 134217729.0

    def split(x):
        t = c * x
        hi = t - (t - x)
        return hi, x - hi

    ah, al = split(a)
    bh, bl = split(b)
    err = ((ah * bh - p) + ah * bl + al * bh) + al * bl
    return math.fsum(np.concatenate([p, err]).tolist())


def dist_setup(a):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v, device="cuda"):
    """Max of a per-rank timing over all ranks (a timing reduce, not data)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(world, ms_local, flop_per_step_per_rank, steps, device="cuda"):
    """Weak scaling: every rank runs its own problem; the job finishes when the
    slowest rank does.  Returns (max ms over ranks, whole-job TFLOP/s)."""
    ms_max = max_over_ranks(world, ms_local, device)
    return ms_max, world * flop_per_step_per_rank * steps / (ms_max / 1e3) / 1e12


# ------------------------------------------------------- pipe peak probes ---
PROBES = (("tcgen05_f16_2sm", "PROBE_F16_2SM", "TFLOP/s"),
          ("tcgen05_f16_1sm", "PROBE_F16_1SM", "TFLOP/s"),
          ("mma_sync_s8", "PROBE_S8_SYNC", "TOPS"))


def pipe_peaks(os2, stream, uuid, target_ms=30.0, reps=5):
    """Throughput ceilings of the tensor-core instructions the library can use,
    from its own self-checking probe kernels (os2_peak_probe): a check run
    (exact result compared on the CUDA cores), then `reps` timed launches of
    about `target_ms` each, CUDA events on the launching stream.  Reported:
    the best and median launch, and the same per SM clock cycle at the median
    sampled SM clock."""
    import torch
    out = {}
    clocks = ClockSampler(uuid)
    time.sleep(0.2)
    for name, const, unit in PROBES:
        kind = getattr(os2, const)
        _, bad, ctas = os2.peak_probe(kind, 64, check=True, stream=stream)
        if os2.get_status(stream):
            raise RuntimeError(f"device status set by the {name} probe")
        # size the launch from a short one
        it0 = 2000
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        os2.peak_probe(kind, it0, stream=stream)
        e0.record(stream)
        os2.peak_probe(kind, it0, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        iters = max(it0, int(it0 * target_ms / max(e0.elapsed_time(e1), 1e-3)))
        rates = []
        for _ in range(reps):
            e0.record(stream)
            fl = os2.peak_probe(kind, iters, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            rates.append(fl / (e0.elapsed_time(e1) / 1e3) / 1e12)
        if os2.get_status(stream):
            raise RuntimeError(f"device status set by the {name} probe")
        out[name] = {"best": max(rates), "median": statistics.median(rates), "unit": unit,
                     "iters": iters, "check_mismatches": bad, "ctas_checked": ctas}
    clk = clocks.stop()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = clk.get("sm_mhz")
    for v in out.values():
        if mhz:
            v["flop_per_sm_cycle_at_median_clock"] = v["median"] * 1e12 / (sms * mhz * 1e6)
    out["clocks"] = clk
    return out


# ------------------------------------------------------------ CPU oracle ---
def oracle_sample(A, Bt, a, seconds, rows_cols=None):
    """Time the oracle on a growing grid of output entries until `seconds`
    of work is reached; returns (entries, elapsed, result)."""
    from oracle import oracle as orc
    mode = orc.FAST if a.mode == "fast" else orc.ACCURATE
    m, n = A.shape[0], Bt.shape[0]
    if rows_cols is not None:
        rows, cols = rows_cols
        t0 = time.perf_counter()
        ref = orc.gemm_entries(A, Bt, a.num_moduli, rows, cols, mode=mode, want_X=False,
                               want_c=False, want_G=False)
        return len(rows) * len(cols), time.perf_counter() - t0, ref, (rows, cols)
    side = 4
    while True:
        rows, cols = workloads.sample_grid(m, n, side, seed=1)
        t0 = time.perf_counter()
        ref = orc.gemm_entries(A, Bt, a.num_moduli, rows, cols, mode=mode, want_X=False,
                               want_c=False, want_G=False)
        dt = time.perf_counter() - t0
        if dt >= seconds * 0.5 or side >= min(m, n):
            return len(rows) * len(cols), dt, ref, (rows, cols)
        grow = math.sqrt(seconds / max(dt, 1e-3))
        side = int(min(min(m, n), max(side * 2, side * min(grow, 8))))


# --------------------------------------------------------------- arms ------
def run_reference(a):
    """The oracle on the host cores: each step is a bounded sample."""
    from oracle import oracle as orc
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    A, Bt = workloads.make_pair("spread", a.m, a.n, a.k, seed=0, phi=a.phi)
    per_step = max(2.0, 120.0 / max(1, a.steps + a.warmup))
    ent, dt, _, rc = oracle_sample(A, Bt, a, per_step)
    for _ in range(a.warmup):
        oracle_sample(A, Bt, a, per_step, rc)
    times = []
    for _ in range(a.steps):
        e, t, _, _ = oracle_sample(A, Bt, a, per_step, rc)
        times.append(t)
    tot = sum(times)
    value = 2.0 * a.k * ent * a.steps / tot / 1e12
    sample = f"{len(rc[0])} rows x {len(rc[1])} columns of C (full k) per step"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * tot / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config(a),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(a):
    import torch

    import rns_emulated_fp64_gb300 as os2
    world, rank, local = dist_setup(a)
    dev = torch.device("cuda", local if world > 1 else 0)
    os2.set_gemm_variant({"tc": os2.GEMM_TC, "tc_1sm": os2.GEMM_TC_1SM, "tc_i8": os2.GEMM_TC_I8,
                          "s8": os2.GEMM_S8_SYNC, "simt": os2.GEMM_SIMT}[a.gemm])
    if a.crt != "default":
        os2.set_crt_variant({"tc": os2.CRT_TC, "simt": os2.CRT_SIMT, "auto": os2.CRT_AUTO}[a.crt])
    m, n, k, N = a.m, a.n, a.k, a.num_moduli
    A, Bt = workloads.make_pair("spread", m, n, k, seed=rank, phi=a.phi)
    Ad = torch.from_numpy(A).to(dev)
    Bd = torch.from_numpy(Bt).to(dev)
    Cd = torch.empty((m, n), dtype=torch.float64, device=dev)
    ws = os2.alloc_workspace(os2.workspace_size(m, n, k, N, a.mode), dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        os2.gemm(Ad, Bd, N, a.mode, out=Cd, workspace=ws, stream=stream)

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    if not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    peaks_probe = None if a.no_peaks else pipe_peaks(os2, stream, uuid)

    for _ in range(a.warmup):
        step()
    st = os2.get_status(stream)
    if st:
        raise RuntimeError(f"device status after warm-up: {os2.status_string(st)}")
    clocks = ClockSampler(uuid)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    os2.profile_start()
    ev0.record(stream)
    for _ in range(a.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    prof = os2.profile_stop()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    st = os2.get_status(stream)
    if st:
        raise RuntimeError(f"device status after timed steps: {os2.status_string(st)}")
    flop = 2.0 * m * n * k
    ms_max, value = aggregate(world, ms, flop, a.steps)

    peaks, src = measured_peaks()
    kern = {}
    for name, (tot, cnt) in prof.items():
        kern[name] = {"launches": cnt, "launches_per_step": cnt / a.steps,
                      "avg_ms": tot / max(cnt, 1), "share": None}
    total_k = sum(v["avg_ms"] * v["launches"] for v in kern.values())
    for v in kern.values():
        v["share"] = v["avg_ms"] * v["launches"] / total_k if total_k else None
    # algorithmic work per step; a step with A in row panels launches steps 3-5
    # once per panel, each launch doing its share
    kp = (k + 63) // 64 * 64
    pb = 1.0 if a.gemm in ("tc_i8", "s8") else 2.0  # bytes per residue in the planes
    algo = {
        "scale": ("GB/s", 8.0 * (m + n) * k),
        "scale_bars": ("GB/s", 8.0 * (m + n) * k + 2.0 * (m + n) * kp),
        "residues": ("GB/s", 8.0 * (m + n) * k + pb * N * (m + n) * kp),
        "gemm_bound": ("TFLOP/s", 2.0 * m * n * k),
        "gemm_modp": ("TFLOP/s", 2.0 * N * m * n * k),
        "crt_unscale": ("GB/s", 1.0 * N * m * n + 8.0 * m * n + 4.0 * (m + n)),
    }
    for name, v in kern.items():
        if name in algo:
            unit, work = algo[name]
            work /= max(v["launches_per_step"], 1.0)
            secs = v["avg_ms"] / 1e3
            if unit == "GB/s":
                v["achieved"] = work / secs / 1e9
                v["unit"] = "GB/s"
                v["frac_of_hbm"] = v["achieved"] / peaks["hbm_gbs"]
            else:
                v["achieved"] = work / secs / 1e12
                v["unit"] = "TFLOP/s"
    g = kern.get("gemm_modp")
    # the burst peak for a timed region shorter than a few seconds, the
    # sustained (power-capped) one for a region that lasts seconds
    timed_s = ms / 1e3
    sustained = timed_s >= 3.0 and "bf16_tflops_sustained" in peaks
    peak_t = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    roofline = None
    work_launch = "N*2mnk / launches per step = %.4g flop" % (
        2.0 * N * m * n * k / max(g["launches_per_step"], 1.0)) if g else None
    if g and a.gemm == "s8" and peaks_probe:
        # the INT8 tensor path outside tcgen05: its own measured peak (MEASURED_PEAKS.json
        # holds no INT8 figure), multiply-adds counted as two operations as in the probe
        s8 = peaks_probe["mma_sync_s8"]["best"]
        roofline = {"bound": "tensor",
                    "kernel": "gemm_modp (mma.sync.m16n8k32 s8 x s8 -> s32, int8 residue planes)",
                    "achieved": g["achieved"], "peak": s8, "unit": "TFLOP/s",
                    "frac": g["achieved"] / s8, "traffic": None,
                    "peak_source": "own mma.sync s8 probe of this run (of measured; int8 "
                                   "operations, multiply-add = 2)",
                    "work_per_launch": work_launch}
    elif g:
        roofline = {"bound": "tensor", "kernel": "gemm_modp (tcgen05.mma kind::f16, FP16-held residues)",
                    "achieved": g["achieved"], "peak": peak_t, "unit": "TFLOP/s",
                    "frac": g["achieved"] / peak_t,
                    "traffic": (kernel_traffic("gemm_modp", f"{m}x{n}x{k}_N{N}_{a.mode}")
                                if a.gemm == "tc" and a.crt == "default" else None),
                    "peak_source": "%s bf16 dense %s (of %s; FP16 rate = BF16 rate); timed region "
                                   "%.2f s" % (src, "sustained" if sustained else "burst", src,
                                               timed_s),
                    "work_per_launch": work_launch}
        if peaks_probe:
            own = peaks_probe["tcgen05_f16_2sm"]["best"]
            roofline["own_pipe_peak"] = {
                "kind_f16_2sm_tflops": own, "frac": g["achieved"] / own,
                "int8_mma_sync_tops": peaks_probe["mma_sync_s8"]["best"],
                "source": "os2_peak_probe, this run (self-checked, operands resident in "
                          "shared memory)"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config(a, {"crt_kernel": a.crt, "gemm_kernel": a.gemm}), "clocks": clk,
            "gpu_launches": os2.launch_count(m, n, k, N, a.mode) * a.steps,
            "roofline": roofline, "kernels": kern}
    if peaks_probe:
        line["pipe_peaks"] = peaks_probe

    # e2e through the host entry point
    if not a.no_e2e:
        Ah = torch.from_numpy(A).pin_memory()
        Bh = torch.from_numpy(Bt).pin_memory()
        Ch = torch.empty((m, n), dtype=torch.float64).pin_memory()
        wsh = os2.alloc_workspace(os2.host_workspace_size(m, n, k, N, a.mode), dev)
        del ws
        torch.cuda.empty_cache()
        for _ in range(3):
            os2.gemm_host(Ah, Bh, Ch, N, a.mode, workspace=wsh, stream=stream)
        torch.cuda.synchronize(dev)
        ke = max(3, a.e2e_calls)
        barrier(world)
        # one event per call as well: the host link is shared with the machine's
        # other tenants, so the spread of single calls is reported beside the mean
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(ke + 1)]
        e0, e1 = evs[0], evs[-1]
        host_ms = []
        e0.record(stream)
        for i in range(ke):
            h0 = time.perf_counter()
            os2.gemm_host(Ah, Bh, Ch, N, a.mode, workspace=wsh, stream=stream)
            host_ms.append(1e3 * (time.perf_counter() - h0))  # enqueue only: the call is async
            evs[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per_call = [evs[i].elapsed_time(evs[i + 1]) for i in range(ke)]
        calls = sorted(per_call)
        barrier(world)
        ems, evalue = aggregate(world, e0.elapsed_time(e1), flop, ke)
        med = calls[len(calls) // 2]
        hmed = sorted(host_ms)[len(host_ms) // 2]
        slow = [{"call": i, "device_ms": per_call[i], "host_enqueue_ms": host_ms[i],
                 "host_enqueue_slow": host_ms[i] > max(5 * hmed, hmed + 1.0)}
                for i in range(ke) if per_call[i] > 1.5 * med]
        trimmed = (sum(per_call) - calls[-1]) / (ke - 1) if ke > 1 else per_call[0]
        line["e2e"] = {"value": evalue, "unit": UNIT,
                       "h2d_bytes_per_step": 8 * (m * k + n * k), "d2h_bytes_per_step": 8 * m * n,
                       "steps": ke, "ms_per_step": ems / ke,
                       "call_ms": {"min": calls[0], "median": med, "max": calls[-1],
                                   "mean": sum(per_call) / ke,
                                   "mean_without_slowest": trimmed,
                                   "tflops_without_slowest": flop / (trimmed / 1e3) / 1e12},
                       "host_enqueue_ms": {"median": hmed, "max": max(host_ms)},
                       "slow_calls": slow}
        assert torch.equal(Ch, Cd.cpu()), "host entry point result differs from device entry point"
        del wsh

    # CPU oracle baseline + bit-exact check of the benchmarked result on the same sample
    if rank == 0 and not a.no_cpu_baseline:
        from oracle import oracle as orc
        ent, dt, ref, (rows, cols) = oracle_sample(A, Bt, a, a.cpu_seconds)
        got = Cd.cpu().numpy()[np.ix_(rows, cols)]
        same = bool(np.array_equal(got.view(np.uint64), ref.C.view(np.uint64)))
        line["cpu_baseline"] = {"value": 2.0 * k * ent / dt / 1e12, "unit": UNIT,
                                "cores": orc.num_threads(), "kind": "oracle",
                                "sample": f"{len(rows)} rows x {len(cols)} columns of C (full k), "
                                          f"{dt:.1f} s",
                                "gpu_result_bit_exact_on_sample": same}
        if not same:
            line["parity_error"] = int(np.count_nonzero(got != ref.C))

    # the metric's INT8 half: the same product with step 3 on the INT8 tensor
    # path (mma.sync s8 on int8 planes), two timed calls; its step-3 rate
    # against this run's mma.sync s8 probe, and its result against the default's
    if not a.no_int8 and a.gemm == "tc":
        ws8 = os2.alloc_workspace(os2.workspace_size(m, n, k, N, a.mode), dev)
        C8 = torch.empty((m, n), dtype=torch.float64, device=dev)
        os2.set_gemm_variant(os2.GEMM_S8_SYNC)
        try:
            os2.gemm(Ad, Bd, N, a.mode, out=C8, workspace=ws8, stream=stream)
            torch.cuda.synchronize(dev)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            os2.profile_start()
            s0.record(stream)
            for _ in range(2):
                os2.gemm(Ad, Bd, N, a.mode, out=C8, workspace=ws8, stream=stream)
            s1.record(stream)
            torch.cuda.synchronize(dev)
            prof8 = os2.profile_stop()
        finally:
            os2.set_gemm_variant(os2.GEMM_TC)
        if os2.get_status(stream):
            raise RuntimeError("device status set during the INT8-path run")
        g8 = prof8.get("gemm_modp")
        ms8 = g8[0] / g8[1]
        tops = 2.0 * N * m * n * k / (g8[1] / 2) / (ms8 / 1e3) / 1e12
        i8 = {"kernel": "k_gemm_s8 (mma.sync.m16n8k32 s8 x s8 -> s32, int8 residue planes)",
              "step3_ms_per_launch": ms8, "step3_tops": tops,
              "emulated_tflops": flop / (s0.elapsed_time(s1) / 2 / 1e3) / 1e12,
              "bit_identical_to_default": bool(torch.equal(C8, Cd))}
        if peaks_probe:
            i8["peak_tops"] = peaks_probe["mma_sync_s8"]["best"]
            i8["frac"] = tops / i8["peak_tops"]
            i8["peak_source"] = "own mma.sync s8 probe of this run (of measured)"
        line["int8_tensor_path"] = i8
        del ws8, C8
        torch.cuda.empty_cache()

    # the rest of the 8192^3 configuration: N in {14, 16, 18}, both modes
    if not a.no_sweep:
        sweep = {}
        for Ns in (14, 16, 18):
            for mode in ("fast", "accurate"):
                wss = os2.alloc_workspace(os2.workspace_size(m, n, k, Ns, mode), dev)
                Cs = torch.empty((m, n), dtype=torch.float64, device=dev)
                for _ in range(2):
                    os2.gemm(Ad, Bd, Ns, mode, out=Cs, workspace=wss, stream=stream)
                torch.cuda.synchronize(dev)
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 10
                s0.record(stream)
                for _ in range(reps):
                    os2.gemm(Ad, Bd, Ns, mode, out=Cs, workspace=wss, stream=stream)
                s1.record(stream)
                torch.cuda.synchronize(dev)
                if os2.get_status(stream):
                    raise RuntimeError("device status set during the sweep")
                sms = s0.elapsed_time(s1) / reps
                sweep[f"N{Ns}_{mode}"] = {"ms": sms, "tflops": flop / (sms / 1e3) / 1e12}
                del wss, Cs
                torch.cuda.empty_cache()
        line["sweep_8192cube"] = sweep
        # SGEMM emulation of the same workload (float32 operands, binary32 result)
        Af, Bf = Ad.float(), Bd.float()
        Cf = torch.empty((m, n), dtype=torch.float32, device=dev)
        wsf = os2.alloc_workspace(os2.workspace_size(m, n, k, 7, "fast"), dev)
        for _ in range(2):
            os2.sgemm(Af, Bf, 7, "fast", out=Cf, workspace=wsf, stream=stream)
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(10):
            os2.sgemm(Af, Bf, 7, "fast", out=Cf, workspace=wsf, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        sms = s0.elapsed_time(s1) / 10
        line["sgemm_8192cube_N7_fast"] = {"ms": sms, "tflops": flop / (sms / 1e3) / 1e12}
        del Af, Bf, Cf, wsf
        torch.cuda.empty_cache()
        # ZGEMM emulation at 4096^3 complex (8mnk real flop), 16 moduli, fast mode
        mz = 4096
        Zr, Zi = workloads.make_pair("spread", mz, mz, mz, seed=rank, phi=a.phi)
        Za = torch.complex(torch.from_numpy(Zr[:, :mz]), torch.from_numpy(Zi[:, :mz])).to(dev)
        Zb = torch.complex(torch.from_numpy(Zi[:, :mz].copy()), torch.from_numpy(Zr[:, :mz].copy())).to(dev)
        wsz = os2.alloc_workspace(os2.complex_workspace_size(mz, mz, mz, 16, "fast"), dev)
        Cz = torch.empty((mz, mz), dtype=torch.complex128, device=dev)
        for _ in range(2):
            os2.zgemm(Za, Zb, 16, "fast", out=Cz, workspace=wsz, stream=stream)
        torch.cuda.synchronize(dev)
        s0.record(stream)
        for _ in range(5):
            os2.zgemm(Za, Zb, 16, "fast", out=Cz, workspace=wsz, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        zms = s0.elapsed_time(s1) / 5
        line["zgemm_4096cube_N16_fast"] = {"ms": zms, "tflops": 8.0 * mz ** 3 / (zms / 1e3) / 1e12}
        del Za, Zb, wsz, Cz
        torch.cuda.empty_cache()

    # context: native cuBLAS DGEMM rate and accuracy against the exact product
    if rank == 0 and not a.no_context:
        Bk = Bd.t()
        torch.matmul(Ad, Bk)
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        Cn = torch.matmul(Ad, Bk)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        nat_ms = t0.elapsed_time(t1)
        rr, cc = workloads.sample_grid(m, n, 16, seed=2)
        ex, scale = exact_products(A, Bt, rr, cc)
        errs = {"native_dgemm": rel_errors(Cn.cpu().numpy()[np.ix_(rr, cc)], ex, scale)}
        errs[f"N{N}_{a.mode}"] = rel_errors(Cd.cpu().numpy()[np.ix_(rr, cc)], ex, scale)
        for Ns in (14, 16, 18):
            if Ns != N:
                wse = os2.alloc_workspace(os2.workspace_size(m, n, k, Ns, a.mode), dev)
                Cs = os2.gemm(Ad, Bd, Ns, a.mode, workspace=wse, stream=stream)
                errs[f"N{Ns}_{a.mode}"] = rel_errors(Cs.cpu().numpy()[np.ix_(rr, cc)], ex, scale)
                del wse, Cs
                torch.cuda.empty_cache()
        line["context"] = {"native_dgemm_tflops": flop / (nat_ms / 1e3) / 1e12,
                           "native_dgemm": "torch.matmul float64 (cuBLAS DGEMM)",
                           "err_over_absprod_max_median": errs,
                           "error_sample": f"{len(rr)}x{len(cc)} entries vs the exact product "
                                           "(Dekker products, fsum)"}
        del Cn
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_peaks_only(a):
    import torch

    import rns_emulated_fp64_gb300 as os2
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    uuid = str(torch.cuda.get_device_properties(0).uuid)
    if not uuid.startswith("GPU-"):
        uuid = "GPU-" + uuid
    peaks, src = measured_peaks()
    out = pipe_peaks(os2, stream, uuid)
    out["measured_peaks_json"] = {"bf16_tflops": peaks.get("bf16_tflops"),
                                  "bf16_tflops_sustained": peaks.get("bf16_tflops_sustained"),
                                  "source": src}
    print(json.dumps({"pipe_peaks": out}), flush=True)


def exact_products(A, Bt, rows, cols):
    """Correctly rounded (AB)_ij and (|A||B|)_ij on a grid of entries."""
    ex = np.array([[exact_dot(A[i], Bt[j]) for j in cols] for i in rows])
    scale = np.abs(A[rows]) @ np.abs(Bt[cols]).T
    return ex, scale


def rel_errors(C, ex, scale):
    r = np.abs(C - ex) / np.where(scale > 0, scale, 1.0)
    return float(r.max()), float(np.median(r))


def run_accuracy(a):
    """Error of the emulated product against the exact one, per config of the
    1024^3 workload, with native cuBLAS DGEMM beside it."""
    import torch

    import rns_emulated_fp64_gb300 as os2
    torch.cuda.set_device(0)
    m = n = k = 1024
    rows, cols = workloads.sample_grid(m, n, 64, seed=1)
    out = {"workload": "1024x1024x1024 FP64, entries (U(0,1)-0.5)*exp(phi*N(0,1)), seed 0",
           "sample": f"{len(rows)} x {len(cols)} entries (seeded grid, last row and column "
                     "included) against the exact product (Dekker products, fsum)",
           "error": "|C_ij - (AB)_ij| / (|A||B|)_ij", "configs": {}}
    for phi in (0.5, 2.0, 4.0):
        A, Bt = workloads.make_pair("spread", m, n, k, seed=0, phi=phi)
        ex, scale = exact_products(A, Bt, rows, cols)
        Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(Bt).cuda()
        nat = torch.matmul(Ad, Bd.t()).cpu().numpy()[np.ix_(rows, cols)]
        mx, md = rel_errors(nat, ex, scale)
        rec = {"native_dgemm": {"max": mx, "median": md}}
        for N in range(12, 21, 2):
            for mode in ("fast", "accurate"):
                C = os2.gemm(Ad, Bd, N, mode).cpu().numpy()[np.ix_(rows, cols)]
                if os2.get_status():
                    raise RuntimeError("device status set")
                mx, md = rel_errors(C, ex, scale)
                rec[f"N{N}_{mode}"] = {"max": mx, "median": md}
        out["configs"][f"phi{phi}"] = rec
    print(json.dumps({"accuracy": out}), flush=True)


def main():
    a = parse()
    if a.accuracy:
        run_accuracy(a)
        return
    if a.peaks_only:
        run_peaks_only(a)
        return
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
