#!/usr/bin/env python
"""Benchmark: GEMM TFLOP/s and % of the bf16 dense peak for the CLC, static-persistent
and non-persistent schedules of the same sm_103a kernel on one GB300 (per rank).

Default workload: M = N = K = 8192, bf16 uniform[-1, 1] (seed 1), fp32 C, 128 x 256 tiles,
cluster 1x1x1.  A "step" is one gemm_run call (one kernel launch over the whole product,
ownership log included).  `value` is the CLC schedule's whole-job throughput; the other
schedules are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--all]

With N > 1 (torchrun, one rank per GPU) every rank runs an independent replica (the
path has no exchange step): weak scaling, max time over ranks.  Replicas create their
handle with multicast off and time no cluster shape that shares operands by TMA
multicast: those kernels run only in a process alone on one GPU.
`--impl reference` times the CPU oracle on the host cores instead (rank 0 only).
The default line also carries `workloads`: the tail sweep at T = 149 and 297, the CTA
pair while an occupier holds 24 SMs, and the grouped problems of equal and of varied
depth, each timed under CLC, static-persistent and non-persistent scheduling with its own
clock record (rank 0 at N = 1 only; `--no-workloads` skips it).
`--all` also runs the whole tail sweep, the CTA-pair run beside an SM occupier and the
grouped problems with traces, and writes them to a JSON file (--all-out, default
bench_all.json).
"""
from __future__ import annotations

import argparse
import hashlib
import re
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

METRIC = "GEMM TFLOP/s & % of bf16 dense peak (CLC vs static vs non-persistent) at 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# files whose change invalidates the committed DRAM-traffic counters
# the device code of the GEMM kernel (the per-shape .cu files only instantiate it; launch
# helpers are host code)
KERNEL_SOURCES = ["kernel.cuh", "ptx.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--all", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload rows of the default line")
    ap.add_argument("--workload-seconds", type=float, default=0.6,
                    help="timed launches per workload row and mode: at least this long (and >= 30 launches)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="--impl reference: CPU seconds for all warm-up and timed steps together")
    ap.add_argument("--settle-ms", type=float, default=0.0,
                    help="untimed back-to-back launches before the first timed mode (a sustained power state)")
    ap.add_argument("--clock-extend-ms", type=float, default=400.0,
                    help="untimed launches after the timed CLC region while the clock sampler runs")
    ap.add_argument("--cooldown-ms", type=float, default=300.0,
                    help="idle time before every timed mode, so each mode (CLC first) starts from the same "
                         "power and clock state")
    ap.add_argument("--out", default=None, help="also append the JSON line to this file")
    ap.add_argument("--all-out", default="bench_all.json", help="where --all writes its JSON")
    ap.add_argument("--all-steps", type=int, default=60)
    ap.add_argument("--workload", default="square", help="square | pair | grouped | grouped_vk | tail<T> | tiny")
    ap.add_argument("--raster-group", type=int, default=16)
    ap.add_argument("--l2-prefetch", type=int, default=-1, help="k-blocks prefetched into L2 (-1: library default)")
    ap.add_argument("--occupy", type=int, default=0, help="SMs held by an occupier kernel while timing")
    ap.add_argument("--trace-modes", action="store_true",
                    help="one traced launch of every timed mode row (\"traced_modes\" in the JSON line)")
    ap.add_argument("--modes", default="clc,static_148,static_sms,nonpersistent,pdl,clusters",
                    help="comma-separated subset of the schedules to time (clc is always first)")
    return ap.parse_args()


# ------------------------------------------------------------------ environment
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed: a comment edit does not
    change the kernel a traffic record was captured on."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


TENSOR_FLOP_PER_SM_CLOCK = 8192   # dense bf16 tcgen05 rate of one SM


def kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blackwell_clc_dynamic_gb300", "csrc")
    for f in KERNEL_SOURCES:
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel_key: str, raster_group: int, l2_prefetch: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source with the same options."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("kernel_hash") != kernel_hash():
        return None
    e = d.get("kernels", {}).get(kernel_key)
    if e is None or e.get("raster_group", 8) != raster_group or e.get("l2_prefetch", 0) != l2_prefetch:
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int, interval_ms: int = 200):
        self.interval_ms = interval_ms
        self.sel = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device)
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                s = str(uuid)
                self.sel = s if s.startswith("GPU-") else "GPU-" + s
        except Exception:
            pass
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms",
               str(self.interval_ms)]
        if self.sel:
            cmd += ["-i", self.sel]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "power_w_max": max(power), "samples": len(sm)}


# ------------------------------------------------------------------ reference arm
def oracle_rows_rate(A, B, rows: int):
    import oracle
    t0 = time.perf_counter()
    oracle.gemm_block(A, B, 0, rows, 0, B.shape[1])
    return time.perf_counter() - t0


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import oracle
    import workloads as wl
    w = wl.SQUARE
    A, B = wl.make_inputs(w)
    t_row = oracle_rows_rate(A, B, 2) / 2
    budget = args.ref_seconds
    rows = max(1, int(budget / max(1, args.steps + args.warmup) / t_row))
    for _ in range(args.warmup):
        oracle.gemm_block(A, B, 0, rows, 0, w.N)
    times = []
    for i in range(args.steps):
        r0 = (i * rows) % (w.M - rows)
        t0 = time.perf_counter()
        oracle.gemm_block(A, B, r0, r0 + rows, 0, w.N)
        times.append(time.perf_counter() - t0)
    flops = 2.0 * rows * w.N * w.K
    total = sum(times)
    value = flops * len(times) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed, "tile": [w.bm, w.bn, 64],
                   "cluster": [1, 1, 1], "sched": "clc", "parallelism": f"replicas x{ws}",
                   "l2": "no flush: operands and C exceed the 129 MB L2",
                   "arm": "CPU oracle (fp64) on the host cores: the pages ship no code to run"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows} rows of C ({rows}x{w.N}x{w.K}) per step, fp64 accumulation"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args)
    return 0


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.out:
        with open(args.out, "a") as f:
            f.write(s + "\n")


# ------------------------------------------------------------------ our arm
def mode_table(cl, bn, planned, sms, ws):
    """One row per timed mode: schedule, static workers, cluster size, B multicast for
    clusters of 2, programmatic dependent launch, ownership log; `sel` names it in --modes.
    "static_148" selects the planned static worker count of the workload's statement (148
    workers, or 74 pairs).  The larger cluster shapes of the same tile sit beside the
    headline, not in it, and only when this process runs alone (ws == 1): their CTAs share
    operand tiles by TMA multicast, which stays out of any run on two or more GPUs."""
    def row(key, sched, sel, nw=0, ccl=None, mcast=0, pdl=0, log=1):
        ccl = cl if ccl is None else ccl
        n = ccl if isinstance(ccl, int) else ccl[0] * ccl[1]
        tma_mcast = n == 4 or (n == 2 and bool(mcast))
        return dict(key=key, sched=sched, sel=sel, nw=nw, cl=ccl, mcast=mcast, pdl=pdl, log=log,
                    tma_multicast=tma_mcast)
    table = [row("clc", "clc", "clc"),
             row(f"static_{planned}", "static", "static_148", nw=planned),
             row("static_sms", "static", "static_sms", nw=sms // cl),
             row("nonpersistent", "nonpersistent", "nonpersistent"),
             row("clc_pdl", "clc", "pdl", pdl=1),
             row("clc_no_log", "clc", "pdl", log=0),
             row("clc_pdl_no_log", "clc", "pdl", pdl=1, log=0)]
    if cl == 1 and bn == 256 and ws == 1:
        table += [row("clc_pair_256x256", "clc", "clusters", ccl=2),
                  row("clc_cluster2_shared_b", "clc", "clusters", ccl=2, mcast=1),
                  row("clc_cluster4_shared_b", "clc", "clusters", ccl=4),
                  row("clc_cluster2x2_shared_ab", "clc", "clusters", ccl=(2, 2, 1))]
    if ws > 1:
        assert not any(r["tma_multicast"] for r in table)
    return table


def time_steps(fn, steps, warmup, stream, barrier, sync):
    import torch
    for _ in range(warmup):
        fn()
    sync()
    barrier()
    sync()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    t1.record(stream)
    sync()
    barrier()
    per = [a.elapsed_time(b) for a, b in ev]
    return t0.elapsed_time(t1), per


def cpu_baseline(A, B, seconds):
    import oracle
    t = oracle_rows_rate(A, B, 4) / 4
    rows = max(4, min(A.shape[0], int(seconds / t)))
    dt = oracle_rows_rate(A, B, rows)
    flops = 2.0 * rows * B.shape[1] * A.shape[1]
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows} of C ({rows}x{B.shape[1]}x{A.shape[1]}), fp64 accumulation, "
                      f"{dt:.1f} s wall"}


def make_case(name):
    """(workload, cluster) for a --workload name."""
    import workloads as wl
    if name == "square":
        return wl.SQUARE, 1
    if name == "pair":
        return wl.PAIR, 2
    if name == "grouped":
        return wl.grouped(), 1
    if name == "grouped_vk":
        return wl.grouped_varied_depth(), 1
    if name.startswith("tail"):
        return wl.tail(int(name[4:])), 1
    if name == "tiny":
        return wl.TINY, 1
    raise SystemExit(f"unknown workload {name}")


def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    import blackwell_clc_dynamic_gb300 as clc
    import workloads as wl

    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))

    def barrier():
        if ws > 1:
            dist.barrier()

    peaks, peaks_src = load_peaks()
    w, cl = make_case(args.workload)
    grouped = bool(w.group_m)
    tile = (w.bm, w.bn, 64)
    if grouped:
        As, Bs = wl.make_inputs(w, pin=True)
        dA = [a.cuda(non_blocking=True) for a in As]
        dB = [b.cuda(non_blocking=True) for b in Bs]
        dC = [torch.empty((m, w.N), dtype=torch.float32, device="cuda") for m in w.group_m]
        A, B = As[0], Bs[0]
    else:
        A, B = wl.make_inputs(w, pin=True)
        dA = A.cuda(non_blocking=True)
        dB = B.cuda(non_blocking=True)
        C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    # with an occupier running, only stream-level synchronisation may be used
    stream = torch.cuda.Stream() if args.occupy else torch.cuda.current_stream()
    # replicas (ws > 1) never load or launch the TMA multicast cluster kernels
    g = clc.Gemm(local, raster_group=args.raster_group, l2_prefetch=args.l2_prefetch, multicast=(ws == 1))
    sms = g.sm_count
    resident = g.max_active_clusters(tile, cl)
    planned = 148 // cl

    def step(mode, nw=0, ccl=None):
        ccl = cl if ccl is None else ccl
        if grouped:
            return lambda: g.run_grouped_v(dA, dB, dC, tile=tile, cluster=ccl, sched=mode, num_workers=nw,
                                           stream=stream)
        return lambda: g.run(dA, dB, C, tile=tile, cluster=ccl, sched=mode, num_workers=nw, stream=stream)

    def sync_all():
        if args.occupy:
            stream.synchronize()
        else:
            torch.cuda.synchronize()

    wanted = set(args.modes.split(",")) | {"clc"}
    order = [r for r in mode_table(cl, w.bn, planned, sms, ws) if r["sel"] in wanted]
    step("clc")()                     # sizes the handle's workspace before any occupier runs
    torch.cuda.synchronize()
    if args.occupy:
        s_occ = torch.cuda.Stream()
        g.occupy_start(args.occupy, limit_ns=120_000_000_000, stream=s_occ)
        g.occupy_wait_resident(10_000)

    # optional settle into a sustained power state before the first mode (--settle-ms)
    t_end = time.perf_counter() + args.settle_ms / 1e3
    settle = step("clc")
    while time.perf_counter() < t_end:
        for _ in range(50):
            settle()
        sync_all()

    modes = {}
    clocks = None
    launches = 0
    kernel_ms = None
    try:
        for r in order:
            key, mode, nw, ccl, mcast, pdl = r["key"], r["sched"], r["nw"], r["cl"], r["mcast"], r["pdl"]
            g.set_opts(cluster_b_multicast=mcast, pdl=pdl, log_enable=r["log"])
            # every mode starts from the same idle state: under the 1.4 kW power cap the clock
            # a mode runs at depends on how long the GPU has been busy before it
            sync_all()
            time.sleep(args.cooldown_ms / 1e3)
            sampler = ClockSampler(local, interval_ms=50) if key == "clc" else None
            if sampler:
                sampler.start()
            total_ms, per = time_steps(step(mode, nw, ccl), args.steps, args.warmup, stream, barrier, sync_all)
            if sampler:
                # a timed region of a few tens of milliseconds may hold no sample: the same
                # launches continue, untimed, until the sampler has seen the load
                fn, t_ext = step(mode, nw, ccl), time.perf_counter() + args.clock_extend_ms / 1e3
                while time.perf_counter() < t_ext:
                    for _ in range(20):
                        fn()
                    sync_all()
                clocks = sampler.stop()
                clocks["window"] = (f"warm-up + {args.steps} timed launches + {args.clock_extend_ms:.0f} ms of the "
                                    f"same launches untimed; nvidia-smi every 50 ms")
            tflops, total_ms = job_throughput(total_ms, args.steps, w.flops, ws)
            modes[key] = {"tflops": tflops, "ms_per_step": total_ms / args.steps,
                          "ms_min": min(per), "ms_median": statistics.median(per), "ms_max": max(per),
                          "pct_bf16_peak_burst": 100.0 * tflops / ws / peaks["bf16_tflops"],
                          "pct_bf16_peak_sustained": 100.0 * tflops / ws / peaks["bf16_tflops_sustained"],
                          "pct_hbm_roofline": 100.0 * w.min_bytes / (total_ms / args.steps * 1e-3) / 1e9
                          / peaks["hbm_gbs"],
                          "workers": nw if mode == "static" else None, "cluster": ccl,
                          "b_multicast": bool(mcast or ccl in (4, (2, 2, 1))), "pdl": bool(pdl), "log": bool(r["log"])}
            if key == "clc":
                launches = args.steps
                kernel_ms = statistics.mean(per)
    finally:
        occ_status = g.occupy_stop() if args.occupy else 0
        g.set_opts(cluster_b_multicast=0, pdl=0, log_enable=1)
    torch.cuda.synchronize()
    g.sync(stream)

    e2e = None
    if not args.no_e2e and not grouped:
        Ch = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
        n_e2e = max(3, min(20, args.steps // 50))

        def e2e_step():
            g.run_host(A, B, Ch, tile=tile, cluster=cl, sched="clc", stream=stream)
        tot, per = time_steps(e2e_step, n_e2e, 5, stream, barrier, torch.cuda.synchronize)
        g.sync(stream)
        tot = max_over_ranks(tot, ws)
        e2e = {"value": ws * n_e2e * w.flops / (tot * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": A.numel() * 2 + B.numel() * 2, "d2h_bytes_per_step": Ch.numel() * 4,
               "steps": n_e2e, "ms_per_step": tot / n_e2e, "api": "gemm_run_host (pinned host buffers)"}

    # one traced launch per schedule (outside the timed region): how evenly the SMs finish
    # and what consuming CLC responses costs
    traced = {}
    traced_modes = None
    if not args.occupy:
        for key, mode, nw in (("clc", "clc", 0), (f"static_{planned}", "static", planned)):
            st = trace_stats(g, step(mode, nw))
            traced[key] = {"launch_span_us": round(st["kernel_span_us"], 1),
                           "sm_last_end_spread_us": round(st["sm_last_end_us"]["max"] - st["sm_last_end_us"]["min"], 1),
                           "producer_wait_for_clc_response_us": st["producer_wait_for_clc_response"],
                           "try_cancel_round_trip_us": st["try_cancel_round_trip"],
                           "epilogue_us_mean": st["epilogue_us"]["mean_us"] if st["epilogue_us"] else None}
        if args.trace_modes:
            traced_modes = {}
            for r in order:
                g.set_opts(cluster_b_multicast=r["mcast"], pdl=r["pdl"], log_enable=r["log"])
                try:
                    traced_modes[r["key"]] = trace_stats(g, step(r["sched"], r["nw"], r["cl"]))
                finally:
                    g.set_opts(cluster_b_multicast=0, pdl=0, log_enable=1)

    if rank != 0:
        g.close()
        if ws > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline and ws == 1:     # the CPU baseline is reported at N = 1 only
        cpu = cpu_baseline(A, B, args.cpu_seconds)

    rows = None
    if not args.no_workloads and ws == 1 and args.workload == "square" and not args.occupy:
        if grouped:
            del dA, dB, dC
        else:
            del dA, dB, C
        torch.cuda.empty_cache()
        rows = workload_rows(g, args, peaks, sms)

    clc_m = modes["clc"]
    achieved = w.flops / (kernel_ms * 1e-3) / 1e12
    kname = f"gemm_kernel<{w.bn},{cl},CLC>"
    l2_pf = args.l2_prefetch if args.l2_prefetch >= 0 else 0   # the library's default distance is 0
    traffic = traffic_for(f"gemm_n{w.bn}_c{cl}_clc_{args.workload}", args.raster_group, l2_pf)
    # the timed unit is one launch of under a millisecond, a kernel timed by itself: its
    # denominator is the burst peak; the sustained fraction is kept beside it for context
    roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
            "peak_kind": f"bf16_tflops, burst ({peaks_src}): each timed step is one launch",
            "frac_of_sustained_peak": achieved / peaks["bf16_tflops_sustained"],
            "sustained_note": "bf16_tflops_sustained is cuBLAS looped for seconds under the power cap",
            "algorithmic_flops_per_launch": w.flops, "algorithmic_min_bytes_per_launch": w.min_bytes,
            "kernel": kname}
    ai = w.flops / w.min_bytes
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if ai < ridge:
        # below the ridge (skinny shapes such as the tail sweep) the HBM roofline binds:
        # algorithmic bytes (each operand read once, C written once) per launch / duration
        gbs = w.min_bytes / (kernel_ms * 1e-3) / 1e9
        roof.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "peak_kind": f"hbm_gbs ({peaks_src})",
                     "tensor_frac_burst": achieved / peaks["bf16_tflops"]})
    roof["arithmetic_intensity"] = ai
    roof["ridge_flop_per_byte"] = ridge
    if not grouped and cl == 1:
        # operand bytes every tile streams from L2 into shared memory (A's 128 x K rows and
        # B's K x 256 columns, bf16), the bound of the one-CTA shape; per launch and per second
        tm, tn = -(-w.M // 128), -(-w.N // w.bn)
        stream = tm * tn * (128 * w.K + w.K * w.bn) * 2.0
        roof["l2_to_smem_operand_bytes_per_launch"] = stream
        roof["l2_to_smem_operand_tbs"] = stream / (kernel_ms * 1e-3) / 1e12
    if clocks and clocks.get("sm_mhz"):
        # the tensor pipe's own bound at the clock the SMs actually ran: 8192 dense bf16 flop
        # per SM clock (one 128 x 256 x 16 MMA per 128 clocks), times the SMs, times the
        # median SM clock sampled during the timed region
        clock_peak = sms * TENSOR_FLOP_PER_SM_CLOCK * clocks["sm_mhz"] * 1e6 / 1e12
        roof["clock_peak"] = clock_peak
        roof["frac_of_clock_peak"] = achieved / clock_peak
    big = w.min_bytes > 129e6
    line = {
        "metric": METRIC, "value": clc_m["tflops"], "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": clc_m["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "fp32",
        "data": "synthetic (seeded bf16, see workloads.py)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "seed": w.seed, "tile": list(tile),
                   "cluster": [cl, 1, 1], "sched": "clc", "parallelism": f"replicas x{ws}",
                   "raster_group": args.raster_group, "l2_prefetch": l2_pf,
                   "occupied_sms": args.occupy,
                   "l2": ("no flush: operands and C exceed the 129 MB L2" if big
                          else "no flush (small case; parity only)"),
                   "sms": sms, "resident_clusters": resident},
        "pct_of_bf16_peak_burst": clc_m["pct_bf16_peak_burst"],
        "pct_of_bf16_peak_sustained": clc_m["pct_bf16_peak_sustained"],
        "modes": modes, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches, "clocks": clocks, "traced_launch": traced,
    }
    if rows is not None:
        line["workloads"] = rows
    if traced_modes is not None:
        line["traced_modes"] = traced_modes
    if args.occupy:
        line["occupier_hit_time_limit"] = bool(occ_status)
    emit(line, args)
    if args.all:
        if rows is None:
            if grouped:
                del dA, dB, dC
            else:
                del dA, dB, C
            torch.cuda.empty_cache()
        run_extras(g, args, peaks, sms)
    g.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def max_over_ranks(x, ws):
    """The slowest rank's value (replicas are timed independently; the job takes as long
    as its slowest replica)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(total_ms_local, steps, flops_per_step, ws):
    """Whole-job TFLOP/s of ws replicas: every rank runs `steps` steps of `flops_per_step`;
    the time is the slowest rank's (weak scaling)."""
    t = max_over_ranks(total_ms_local, ws)
    return ws * steps * flops_per_step / (t * 1e-3) / 1e12, t


# ------------------------------------------------------------------ workload rows of the default line
def time_for(fn, stream, seconds, min_steps=30, warmup=5, max_steps=20000):
    """Per-launch CUDA-event times (ms) of a loop on `stream` that lasts at least `seconds`
    (and at least `min_steps` launches), after `warmup` untimed launches; only `stream` is
    synchronised (an SM occupier may hold other SMs meanwhile)."""
    import torch
    for _ in range(warmup):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        fn()
    b.record(stream)
    stream.synchronize()
    est = max(a.elapsed_time(b) / 5, 1e-3)
    steps = int(min(max_steps, max(min_steps, math.ceil(seconds * 1e3 / est))))
    return time_stream(fn, steps, 0, stream)


def workload_rows(g, args, peaks, sms):
    """The workloads the statement quotes beside the square, each under CLC, static-persistent
    (the statement's 148 workers or 74 pairs, and the queried SM count) and non-persistent
    scheduling: the tail sweep at T = 149 and 297 (one tile more than a wave of 148 planned
    workers), CTA pairs while an occupier holds 24 SMs, the grouped problems of equal depth
    and of varied depth.  Every (workload, schedule) pair is one timed loop with its own
    nvidia-smi clock record."""
    import torch

    import workloads as wl

    st = torch.cuda.Stream()
    out = {}

    def timed(label, fn, flops, min_bytes, extra=None):
        st.synchronize()
        time.sleep(args.cooldown_ms / 1e3)   # the same idle state before every loop
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        try:
            per = time_for(fn, st, args.workload_seconds)
        finally:
            clocks = sampler.stop()
        r = summarise(per, flops, min_bytes, peaks)
        r.update({"launches": len(per), "clocks": clocks})
        if extra:
            r.update(extra)
        return r

    def ratios(row, static_key):
        m = row["modes"]
        row["clc_speedup_vs_" + static_key] = m[static_key]["ms_mean"] / m["clc"]["ms_mean"]
        row["clc_speedup_vs_nonpersistent"] = m["nonpersistent"]["ms_mean"] / m["clc"]["ms_mean"]

    # tail sweep: 128 x 256 tiles, T tiles; A alone (T x 2 MiB) exceeds L2, no flush needed
    resident = g.max_active_clusters((128, 256, 64), 1)
    for T in (149, 297):
        w = wl.tail(T)
        A, B = wl.make_inputs(w)
        dA, dB = A.cuda(), B.cuda()
        C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        row = {"workload": w.name, "tiles": T, "resident_workers": resident, "modes": {},
               "l2": "no flush: A exceeds the 129 MB L2"}
        for key, mode, nw in (("clc", "clc", 0), ("static_148", "static", 148), ("static_sms", "static", sms),
                              ("nonpersistent", "nonpersistent", 0)):
            row["modes"][key] = timed(key, lambda: g.run(dA, dB, C, sched=mode, num_workers=nw, stream=st),
                                      w.flops, w.min_bytes, {"workers": nw or None})
        ratios(row, "static_148")
        out[f"tail_T{T}"] = row
        del dA, dB, C
        torch.cuda.empty_cache()

    # CTA pairs (256 x 256 cluster tiles) while 24 SMs are held by the occupier
    w = wl.PAIR
    A, B = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    del A, B
    pair_modes = (("clc", "clc", 0), ("static_74", "static", 74), ("static_sms", "static", sms // 2),
                  ("nonpersistent", "nonpersistent", 0))
    for key, mode, nw in pair_modes:   # sizes the handle's log before the occupier runs
        g.run(dA, dB, C, cluster=2, sched=mode, num_workers=nw, stream=st)
    torch.cuda.synchronize()
    row = {"workload": w.name + "_occupied24", "cluster_tiles": (w.M // 256) * (w.N // 256),
           "resident_pairs_unoccupied": g.max_active_clusters((128, 256, 64), 2), "occupied_sms": 24,
           "free_pairs": (sms - 24) // 2, "modes": {}}
    so = torch.cuda.Stream()
    g.occupy_start(24, limit_ns=60_000_000_000, stream=so)
    try:
        g.occupy_wait_resident(10_000)
        for key, mode, nw in pair_modes:
            row["modes"][key] = timed(key, lambda: g.run(dA, dB, C, cluster=2, sched=mode, num_workers=nw,
                                                         stream=st), w.flops, w.min_bytes, {"workers": nw or None})
    finally:
        row["occupier_hit_time_limit"] = bool(g.occupy_stop())
    torch.cuda.synchronize()
    ratios(row, "static_74")
    out["pair_occupied24"] = row
    del dA, dB, C
    torch.cuda.empty_cache()

    # grouped problems: equal depth (K = 4096), then varied depth (K_g)
    for label, w in (("grouped", wl.grouped()), ("grouped_varied_depth", wl.grouped_varied_depth())):
        As, Bs = wl.make_inputs(w)
        dA = [a.cuda() for a in As]
        dB = [b.cuda() for b in Bs]
        del As, Bs
        dC = [torch.empty((m, w.N), dtype=torch.float32, device="cuda") for m in w.group_m]
        torch.cuda.synchronize()
        row = {"workload": w.name, "problems": len(w.group_m),
               "tiles": sum((m // 128) * (w.N // 256) for m in w.group_m), "modes": {}}
        if w.group_k:
            row["k_min"], row["k_max"] = min(w.group_k), max(w.group_k)
        for key, mode, nw in (("clc", "clc", 0), ("static_148", "static", 148), ("static_sms", "static", sms),
                              ("nonpersistent", "nonpersistent", 0)):
            row["modes"][key] = timed(key, lambda: g.run_grouped_v(dA, dB, dC, sched=mode, num_workers=nw,
                                                                   stream=st), w.flops, w.min_bytes,
                                      {"workers": nw or None})
        ratios(row, "static_148")
        out[label] = row
        del dA, dB, dC
        torch.cuda.empty_cache()
    g.sync(st)
    return out


# ------------------------------------------------------------------ --all: the other workloads
def time_stream(fn, steps, warmup, stream):
    """Per-step CUDA-event times on `stream`, synchronising only that stream (an SM
    occupier may be running on another one)."""
    import torch
    for _ in range(warmup):
        fn()
    stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_stream_flushed(fn, steps, warmup, stream, flush):
    """Like time_stream, but L2 is flushed (a buffer larger than L2 is overwritten) before
    every timed launch; the flush lies outside the timed events."""
    import torch
    for _ in range(warmup):
        fn()
    stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        with torch.cuda.stream(stream):
            flush.add_(1)
        a.record(stream)
        fn()
        b.record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def summarise(per_ms, flops, min_bytes, peaks):
    med = statistics.median(per_ms)
    mean = statistics.mean(per_ms)
    tf = flops / (mean * 1e-3) / 1e12
    return {"tflops": tf, "ms_mean": mean, "ms_median": med, "ms_min": min(per_ms), "ms_max": max(per_ms),
            "pct_bf16_peak_burst": 100 * tf / peaks["bf16_tflops"],
            "pct_hbm_roofline": 100 * (min_bytes / (mean * 1e-3) / 1e9) / peaks["hbm_gbs"]}


def trace_stats(g, run_once):
    """One traced run: per-tile CLC waits and round trips, per-SM active span.  Only the
    run's own stream is synchronised (an occupier may hold other SMs meanwhile); the
    trace buffer must already be large enough (a traced run of the same size happened
    before any occupier started), since growing it synchronises the device."""
    g.set_opts(trace_enable=1)
    try:
        run_once()
        tr = g.get_trace().astype(np.int64)
    finally:
        g.set_opts(trace_enable=0)
    start, end, sm = tr[:, 0], tr[:, 1], tr[:, 2]
    ok = (start > 0) & (end > 0)
    t0 = start[ok].min()
    span = {}
    for s_, e_, m_ in zip(start[ok], end[ok], sm[ok]):
        a, b = span.get(int(m_), (s_, e_))
        span[int(m_)] = (min(a, s_), max(b, e_))
    busy = np.array([b - a for a, b in span.values()], dtype=np.float64)
    last = np.array([b - t0 for a, b in span.values()], dtype=np.float64)
    wait = tr[:, 4][tr[:, 4] > 0].astype(np.float64)
    rt = tr[:, 5][tr[:, 5] > 0].astype(np.float64)
    epi_ok = ok & (tr[:, 6] > 0)
    epilogue = (end[epi_ok] - tr[epi_ok, 6]).astype(np.float64)
    main_ok = ok & (tr[:, 7] > 0)
    mainloop = (tr[main_ok, 7] - start[main_ok]).astype(np.float64)

    def q(x):
        if x.size == 0:
            return None
        return {"n": int(x.size), "mean_us": float(x.mean() / 1e3), "p50_us": float(np.percentile(x, 50) / 1e3),
                "p99_us": float(np.percentile(x, 99) / 1e3), "max_us": float(x.max() / 1e3)}
    return {"sms_used": len(span), "kernel_span_us": float((end[ok].max() - t0) / 1e3),
            "sm_active_span_us": {"min": float(busy.min() / 1e3), "mean": float(busy.mean() / 1e3),
                                  "max": float(busy.max() / 1e3)},
            "sm_last_end_us": {"min": float(last.min() / 1e3), "max": float(last.max() / 1e3)},
            "tile_us": q((end[ok] - start[ok]).astype(np.float64)),
            "producer_wait_for_clc_response": q(wait), "try_cancel_round_trip": q(rt),
            "epilogue_us": q(epilogue), "start_to_last_mma_us": q(mainloop)}


def run_extras(g, args, peaks, sms):
    import torch

    import workloads as wl

    out = {"peaks": peaks, "sms": sms, "steps": args.all_steps, "tail": [], "pair": {}, "grouped": {}}
    steps, warm = args.all_steps, 5
    st = torch.cuda.Stream()

    # tail sweep: M = 128 T, N = 256, K = 8192 (seed 2): CLC vs static, with and without an
    # L2 flush (256 MiB write) before every timed launch
    resident = g.max_active_clusters((128, 256, 64), 1)
    flush = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")
    for T in wl.TAIL_T:
        w = wl.tail(T)
        A, B = wl.make_inputs(w)
        dA, dB = A.cuda(), B.cuda()
        C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        row = {"workload": w.name, "T": T, "tiles": T, "resident": resident,
               "model_waves": {"clc": math.ceil(T / resident), "static_148": math.ceil(T / 148)}}
        for key, mode, nw in (("clc", "clc", 0), ("static_148", "static", 148), ("static_sms", "static", sms)):
            per = time_stream(lambda: g.run(dA, dB, C, sched=mode, num_workers=nw, stream=st), steps, warm, st)
            row[key] = summarise(per, w.flops, w.min_bytes, peaks)
            per = time_stream_flushed(lambda: g.run(dA, dB, C, sched=mode, num_workers=nw, stream=st), steps, warm,
                                      st, flush)
            row[key]["l2_flushed"] = summarise(per, w.flops, w.min_bytes, peaks)
            if T in (149, 297) and key != "static_sms":
                row[key]["trace"] = trace_stats(g, lambda: g.run(dA, dB, C, sched=mode, num_workers=nw, stream=st))
        out["tail"].append(row)
        del dA, dB, C
        torch.cuda.empty_cache()
    del flush

    # a higher-priority kernel that cannot share an SM with the GEMM arrives while a CLC
    # GEMM runs: cancels may fail early (the pages' second failure cause); count the
    # workers that ran and how many tiles each took
    w = wl.tail(152 * 8)
    A, B = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    del A, B
    lo, hi = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1)
    g.run(dA, dB, C, stream=lo)
    torch.cuda.synchronize()
    prio = {"workload": w.name, "tiles": w.M // 128, "occupier_ctas": 24}
    for label, occupy in (("alone", False), ("occupier_at_higher_priority", True)):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(lo)
        g.run(dA, dB, C, stream=lo)
        ev1.record(lo)
        if occupy:
            g.occupy_start(24, limit_ns=20_000_000_000, stream=hi)
        try:
            lo.synchronize()
        finally:
            status = g.occupy_stop() if occupy else 0
        torch.cuda.synchronize()
        owner, claims, first = g.get_log()
        counts = np.bincount(owner)
        prio[label] = {"ms": ev0.elapsed_time(ev1), "workers_ran": int((first >= 0).sum()),
                       "max_tiles_per_worker": int(counts.max()), "min_tiles_per_worker": int(counts[counts > 0].min()),
                       "claims_exactly_once": bool((claims == 1).all()), "occupier_hit_limit": bool(status)}
    out["priority"] = prio
    del dA, dB, C
    torch.cuda.empty_cache()

    # CTA pairs while 24 SMs are held by an occupier on another stream
    w = wl.PAIR
    A, B = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
    del A, B
    torch.cuda.synchronize()
    tiles = (w.M // 256) * (w.N // 256)
    res_pairs = g.max_active_clusters((128, 256, 64), 2)
    pair = {"workload": w.name, "cluster_tiles": tiles, "resident_pairs_unoccupied": res_pairs}
    modes = (("clc", "clc", 0), ("static_74", "static", 74), ("static_sms", "static", sms // 2),
             ("nonpersistent", "nonpersistent", 0))
    for occupied in (False, True):
        so = torch.cuda.Stream()
        res = {}
        if occupied:
            g.occupy_start(24, limit_ns=60_000_000_000, stream=so)
            g.occupy_wait_resident(10_000)
        try:
            for key, mode, nw in modes:
                per = time_stream(lambda: g.run(dA, dB, C, cluster=2, sched=mode, num_workers=nw, stream=st),
                                  steps, warm, st)
                res[key] = summarise(per, w.flops, w.min_bytes, peaks)
                if key in ("clc", "static_74"):
                    res[key]["trace"] = trace_stats(
                        g, lambda: g.run(dA, dB, C, cluster=2, sched=mode, num_workers=nw, stream=st))
        finally:
            status = g.occupy_stop() if occupied else 0
        torch.cuda.synchronize()
        res["occupier_hit_time_limit"] = bool(status)
        res["free_pairs"] = (sms - (24 if occupied else 0)) // 2
        pair["occupied_24_sms" if occupied else "all_sms"] = res
    out["pair"] = pair
    del dA, dB, C
    torch.cuda.empty_cache()

    # grouped: 64 problems in one flat grid
    w = wl.grouped()
    As, Bs = wl.make_inputs(w)
    dA = [a.cuda() for a in As]
    dB = [b.cuda() for b in Bs]
    del As, Bs
    dC = [torch.empty((m, w.N), dtype=torch.float32, device="cuda") for m in w.group_m]
    torch.cuda.synchronize()
    grp = {"workload": w.name, "problems": len(w.group_m), "rows": sum(w.group_m),
           "tiles": sum(m // 128 for m in w.group_m) * (w.N // 256)}
    for key, mode, nw in (("clc", "clc", 0), ("static_148", "static", 148), ("static_sms", "static", sms),
                          ("nonpersistent", "nonpersistent", 0)):
        per = time_stream(lambda: g.run_grouped(dA, dB, dC, sched=mode, num_workers=nw, stream=st), steps, warm, st)
        grp[key] = summarise(per, w.flops, w.min_bytes, peaks)
        if key in ("clc", "static_148"):
            grp[key]["trace"] = trace_stats(g, lambda: g.run_grouped(dA, dB, dC, sched=mode, num_workers=nw,
                                                                     stream=st))
    out["grouped"] = grp
    g.sync(st)
    del dA, dB, dC
    torch.cuda.empty_cache()

    # grouped problems of different depth: tiles of unequal cost
    w = wl.grouped_varied_depth()
    As, Bs = wl.make_inputs(w)
    dA = [a.cuda() for a in As]
    dB = [b.cuda() for b in Bs]
    del As, Bs
    dC = [torch.empty((m, w.N), dtype=torch.float32, device="cuda") for m in w.group_m]
    torch.cuda.synchronize()
    T = sum((m // 128) * (w.N // 256) for m in w.group_m)
    vk = {"workload": w.name, "problems": len(w.group_m), "rows": sum(w.group_m), "tiles": T,
          "k_min": min(w.depths()), "k_max": max(w.depths())}
    for key, mode, nw in (("clc", "clc", 0), ("static_148", "static", 148), ("static_sms", "static", sms),
                          ("nonpersistent", "nonpersistent", 0)):
        per = time_stream(lambda: g.run_grouped_v(dA, dB, dC, sched=mode, num_workers=nw, stream=st), steps, warm,
                          st)
        vk[key] = summarise(per, w.flops, w.min_bytes, peaks)
        if key in ("clc", "static_148"):
            vk[key]["trace"] = trace_stats(g, lambda: g.run_grouped_v(dA, dB, dC, sched=mode, num_workers=nw,
                                                                      stream=st))
    # how far ahead a worker may fetch (the throttle): extra tiles held in reserve
    vk["fetch_ahead"] = {}
    for ahead in (0, 1, 2):
        g.set_opts(fetch_ahead=ahead)
        per = time_stream(lambda: g.run_grouped_v(dA, dB, dC, sched="clc", stream=st), steps, warm, st)
        vk["fetch_ahead"][str(ahead)] = summarise(per, w.flops, w.min_bytes, peaks)
        vk["fetch_ahead"][str(ahead)]["trace"] = trace_stats(
            g, lambda: g.run_grouped_v(dA, dB, dC, sched="clc", stream=st))
    g.set_opts(fetch_ahead=0)
    out["grouped_varied_depth"] = vk
    g.sync(st)

    path = args.all_out
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(f"# --all results written to {path}", file=sys.stderr)


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
