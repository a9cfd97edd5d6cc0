#!/usr/bin/env python
"""Benchmark of the fused 3x3(x3) convolution hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--path auto|tc|fma] [--no-others]

One step = one conv3d_fused call (valid 3x3x3 conv with the fused epilogue) over
one batch of seeded synthetic input already resident in HBM.  The default
workload is conv3d + tanh(mish) on x[16,32,32,64,64] -> [16,64,30,62,62].
Prints ONE JSON line on rank 0.  Under torchrun each rank runs its own batch
shard on its own GPU (weak scaling; the only collectives are the timing
barrier and the max over ranks).

--impl reference times the float64 CPU oracle (the checker) on the host cores,
each step a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "conv GFLOP/s (2·MACs/time), µs/call, % of fp32/TF32 or HBM roofline"
UNIT = "GFLOP/s"
L2_BYTES = 129 * 1024 * 1024
# Nominal dense tensor rates (PFLOP/s): TF32 / BF16 ratio used to derive the TF32 peak
# from the measured BF16 GEMM rate.
TF32_OVER_BF16 = 1.1 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
SMS = 152
FMA_PER_SM_PER_CLK = 128

WORKLOADS = {
    "conv3d_tanh_mish": si.conv3d_tanh_mish,
    "conv3d_pool_reduce": si.conv3d_pool_reduce,
    "dwsep": si.dwsep_conv2d,
    "sweep16": lambda: si.conv3d_sweep(16),
    "sweep64": lambda: si.conv3d_sweep(64),
    "sweep128": lambda: si.conv3d_sweep(128),
    "tiny": si.tiny_conv3d,
    "conv3d_same": si.conv3d_same_tanh_mish,
    "conv3d_s2": si.conv3d_stride2_tanh_mish,
    "dwsep_k5": si.dwsep_k5,
}


def with_batch(wl, n: int):
    """The same workload with batch size n (same seed and distributions)."""
    import dataclasses
    tensors = [dataclasses.replace(t, shape=(n,) + tuple(t.shape[1:])) if t.name == "x" else t
               for t in wl.tensors]
    return dataclasses.replace(wl, name=f"{wl.name}_batch{n}", tensors=tensors)


# ------------------------------------------------------------------ workload arithmetic
def conv_out_dims(wl) -> tuple:
    d, p, s = wl.dims, wl.pad, wl.stride
    return tuple((d[k] + 2 * p - 3) // s + 1 for k in ("D", "H", "W"))


def macs(wl) -> int:
    d = wl.dims
    if wl.op == "conv3d":
        od, oh, ow = conv_out_dims(wl)
        return d["N"] * d["Cout"] * od * oh * ow * d["Cin"] * 27
    return d["N"] * d["H"] * d["W"] * d["C"] * (d["K"] * d["K"] + d["Cout"])


def compulsory_bytes(wl) -> tuple:
    """(bytes read, bytes written) if every input is read once and every output written once."""
    rd = sum(t.numel for t in wl.tensors) * 4
    d = wl.dims
    if wl.op == "conv3d":
        if wl.epilogue == "pool_reduce":
            wr = d["N"] * 4
        else:
            od, oh, ow = conv_out_dims(wl)
            wr = d["N"] * d["Cout"] * od * oh * ow * 4
    else:
        wr = d["N"] * d["Cout"] * d["H"] * d["W"] * 4
    return rd, wr


def describe(wl) -> str:
    d = wl.dims
    if wl.op == "conv3d":
        epi = {"tanh_mish": "tanh(mish)", "pool_reduce": "/2-maxpool2-mean-+bias2-sum_c",
               "none": "none"}[wl.epilogue]
        kind = f"pad{wl.pad}" if wl.pad else "valid"
        return (f"conv3d k3 {kind} s{wl.stride} x[{d['N']},{d['Cin']},{d['D']},{d['H']},{d['W']}] "
                f"w[{d['Cout']},{d['Cin']},3,3,3] epilogue {epi}")
    return (f"dwsep conv2d x[{d['N']},{d['C']},{d['H']},{d['W']}] dw {d['K']}x{d['K']} pad{(d['K'] - 1) // 2} -> pw "
            f"{d['C']}->{d['Cout']}, no bias")


def load_peaks() -> tuple:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def roofline_peak(path: str, op: str, peaks: dict, src: str) -> dict:
    """The roofline the dominant kernel of a path is held to."""
    if path == "tc" and op == "conv3d":
        tf32 = peaks["bf16_tflops"] * TF32_OVER_BF16
        return {"bound": "tensor", "peak": tf32 / 3.0, "unit": "TFLOP/s",
                "peak_note": (f"3xTF32: dense TF32 peak / 3; TF32 = {src} BF16 GEMM burst "
                              f"{peaks['bf16_tflops']:.0f} TFLOP/s x nominal TF32/BF16 ratio 1.1/2.25")}
    if path == "tc":
        return {"bound": "hbm", "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_note": f"{src} HBM copy bandwidth"}
    mhz = peaks.get("sm_max_mhz", 2070.0)
    fma_tf = SMS * FMA_PER_SM_PER_CLK * 2 * mhz * 1e6 / 1e12
    return {"bound": "alu", "peak": fma_tf, "unit": "TFLOP/s",
            "peak_note": f"FP32 FMA: {SMS} SMs x {FMA_PER_SM_PER_CLK} FMA/clk x 2 FLOP x {mhz:.0f} MHz"}


def traffic_for(kernel_key: str, wl_name: str):
    """ncu DRAM bytes per launch recorded under profiles/, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(kernel_key, {}).get(wl_name)
    except (OSError, ValueError):
        return None
    if not rec or not rec.get("sources") or not rec.get("sources_sha256"):
        return None
    return rec["dram_bytes_per_launch"] if sources_sha256(rec["sources"]) == rec["sources_sha256"] else None


def sources_sha256(paths):
    """sha256 over the named source files, in order (None if one is missing)."""
    h = hashlib.sha256()
    try:
        for rel in paths:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return h.hexdigest() if paths else None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for t, r in self.samples if t0 <= t <= t1 + 0.15]
        if not rows:
            rows = [r for _, r in self.samples[-3:]]
        mhz, mx, reasons = [], [], set()
        for r in rows:
            try:
                mhz.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(self.NAMES, r[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


# ------------------------------------------------------------------ our arm
def shard_inputs(wl, rank: int, world: int) -> dict:
    """Inputs of this rank: batch items [rank*N, (rank+1)*N) of a global batch of N*world."""
    out = {}
    x = wl.spec("x")
    shard_numel = x.numel
    global_x = x.numel * world
    off = 0
    for t in wl.tensors:
        if t.name == "x":
            out["x"] = si.draw(wl.seed, rank * shard_numel, t.shape, t.dist)
            off = global_x
        else:
            out[t.name] = si.draw(wl.seed, off, t.shape, t.dist)
            off += t.numel
    return out


def make_call(ig3, wl, dev_t: dict, path: str):
    import torch
    if wl.op == "conv3d":
        d = wl.dims
        params = None
        if wl.epilogue == "pool_reduce":
            params = {"divisor": wl.divisor, "pool": wl.pool, "bias2": dev_t["bias2"]}
            out = torch.empty((d["N"],), device=dev_t["x"].device)
        else:
            out = torch.empty((d["N"], d["Cout"]) + conv_out_dims(wl), device=dev_t["x"].device)
        p2 = 2 * wl.pad
        if wl.stride == 1:
            need = ig3.conv3d_fused_pad_workspace_size(d["N"], d["Cin"], d["D"], d["H"], d["W"], wl.pad, d["Cout"],
                                                       wl.epilogue, path)
            chosen = ig3.conv3d_fused_select_path(d["N"], d["Cin"], d["D"] + p2, d["H"] + p2, d["W"] + p2,
                                                  d["Cout"], wl.epilogue, path)
        else:
            # strided: the tensor-core kernel (its split weights in the workspace) where
            # it applies, else the FMA kernel (no workspace)
            need = ig3.conv3d_fused_ex_workspace_size(d["N"], d["Cin"], d["D"], d["H"], d["W"], wl.pad, wl.stride,
                                                      d["Cout"], wl.epilogue, path)
            chosen = "tc" if need > 0 else "fma"
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev_t["x"].device)

        def call():
            ig3.conv3d_fused(dev_t["x"], dev_t["w"], dev_t.get("b"), epilogue=wl.epilogue, params=params, out=out,
                             workspace=ws, path=path, pad=wl.pad, stride=wl.stride)
        return call, out, chosen
    d = wl.dims
    out = torch.empty((d["N"], d["Cout"], d["H"], d["W"]), device=dev_t["x"].device)
    chosen = ig3.dwsep_conv2d_ex_select_path(d["N"], d["C"], d["H"], d["W"], d["K"], d["Cout"], path)

    def call():
        ig3.dwsep_conv2d(dev_t["x"], dev_t["w_dw"], dev_t["w_pw"], dev_t.get("b"), out=out, path=path)
    return call, out, chosen


def time_steps(call, steps: int, warmup: int, dist_on: bool):
    import torch
    import torch.distributed as dist
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if dist_on:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record()
    for _ in range(steps):
        call()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if dist_on:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(end), dist_on)
    return ms, t0, t1


def max_over_ranks(value: float, dist_on: bool, device: str = "cuda") -> float:
    """The largest `value` over all ranks: the job takes as long as its slowest rank."""
    if not dist_on:
        return value
    import torch
    import torch.distributed as dist
    v = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(v, op=dist.ReduceOp.MAX)
    return float(v.item())


def job_gflops(flop_per_rank: float, world: int, us_per_step: float) -> float:
    """Whole-job throughput: the work of every rank over the (slowest rank's) step time."""
    return flop_per_rank * world / (us_per_step * 1e-6) / 1e9


def e2e_steps(ig3, wl, path: str, dev_t: dict, steps: int, warmup: int):
    """The public call with each step's inputs copied from pinned host memory and its output
    read back into pinned host memory, as a serving loop runs it: two device buffer sets,
    one stream each for uploads, the call and downloads, ordered by events, so step i+1's
    upload and step i-1's download overlap step i's compute.  Every step's copies are
    inside the timed region.  Returns (ms for `steps` steps, h2d bytes/step, d2h bytes/step)."""
    import torch
    host = {k: v.cpu().pin_memory() for k, v in dev_t.items()}
    sets = []
    for _ in range(2):
        dt = {k: torch.empty_like(v) for k, v in dev_t.items()}
        call, out, _ = make_call(ig3, wl, dt, path)
        sets.append((dt, call, out, torch.empty(out.shape, dtype=out.dtype).pin_memory()))
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        b = i & 1
        dt, call, out, out_host = sets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_run[b])       # buffer b's inputs are free once its last call ran
            for k, v in host.items():
                dt[k].copy_(v, non_blocking=True)
            ev_in[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev_in[b])
            if used[b]:
                s_run.wait_event(ev_out[b])      # and its output once it was read back
            call()
            ev_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_run[b])
            out_host.copy_(out, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        step(warmup + i)
    s_out.wait_event(ev_out[(warmup + steps - 1) & 1])
    end.record(s_out)
    torch.cuda.synchronize()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sets[0][3].numel() * sets[0][3].element_size()
    return start.elapsed_time(end), h2d, d2h


def host_link_peaks(nbytes: int = 256 << 20) -> dict:
    """Pinned host <-> device copy bandwidth on this machine (GB/s): each direction alone and
    both at once on two streams (best of 5, CUDA events), the ceiling of the end-to-end
    pipeline's copies."""
    import torch
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        best = float("inf")
        for _ in range(5):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d_a.copy_(h_src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)

    def both():
        h2d()
        d2h()
    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": round(nbytes / t_h2d / 1e9, 1), "d2h_gbs": round(nbytes / t_d2h / 1e9, 1),
            "concurrent_gbs": round(2 * nbytes / t_both / 1e9, 1),
            "how": "pinned 256 MiB copies, best of 5, host wall clock around a synchronised copy"}


def measure_workload(ig3, wl, path, steps, warmup, peaks, src, rank=0, world=1, dist_on=False, clocks=None):
    import torch
    t = shard_inputs(wl, rank, world)
    dev_t = {k: torch.from_numpy(v).cuda() for k, v in t.items()}
    call, out, chosen = make_call(ig3, wl, dev_t, path)
    launches0 = ig3.ig3_kernel_launches()
    ms, t0, t1 = time_steps(call, steps, warmup, dist_on)
    launches = ig3.ig3_kernel_launches() - launches0
    if ig3.ig3_last_device_status() != 0:
        raise RuntimeError("a kernel reported a device-side timeout during the benchmark")
    per_step_launches = launches // (steps + warmup) if steps + warmup else 0
    flop = 2.0 * macs(wl)
    us = ms * 1e3 / steps
    gflops = job_gflops(flop, world, us)
    roof = roofline_peak(chosen, wl.op, peaks, src)
    if roof["unit"] == "GB/s":
        rd, wr = compulsory_bytes(wl)
        achieved = (rd + wr) / (us * 1e-6) / 1e9
    else:
        achieved = flop / (us * 1e-6) / 1e12
    res = {"workload": wl.name, "path": chosen, "us_per_call": us, "gflops": gflops, "ms_total": ms,
           "timed_launches": per_step_launches * steps, "launches_per_call": per_step_launches,
           "roofline": {"bound": roof["bound"], "achieved": achieved, "peak": roof["peak"], "unit": roof["unit"],
                        "frac": achieved / roof["peak"], "peak_note": roof["peak_note"]},
           "t0": t0, "t1": t1, "dev_t": dev_t, "call": call, "out": out}
    return res


def oracle_sample(wl, target_s: float):
    """A bounded sample of the workload for the oracle, sized to take about target_s.

    Returns (run, flop, description): run() executes the oracle on the sample and
    returns its wall time in seconds; flop is the sample's algorithmic FLOP count.
    """
    import oracle
    t = shard_inputs(wl, 0, 1)
    d = wl.dims
    if wl.op == "conv3d":
        _, oh, ow = conv_out_dims(wl)

        def make(planes, items=1):
            # input planes that the first `planes` output planes read (the slab's far
            # end then reads the zero border: the same work, for timing)
            xs = np.ascontiguousarray(t["x"][0:items, :, 0:max(1, (planes - 1) * wl.stride + 3 - 2 * wl.pad)])

            def run():
                t0 = time.perf_counter()
                y = oracle.conv3d_ex(xs, t["w"], t.get("b"), wl.pad, wl.stride)
                if wl.epilogue == "tanh_mish":
                    oracle.tanh_mish(y)
                elif wl.epilogue == "pool_reduce":
                    oracle.pool_reduce(y, wl.divisor, wl.pool, t["bias2"])
                return time.perf_counter() - t0
            return run, 2.0 * items * d["Cout"] * planes * oh * ow * d["Cin"] * 27
        one, _ = make(2)
        dt = one()
        od = conv_out_dims(wl)[0]
        planes = int(max(2, min(od, 2 * target_s / max(dt, 1e-3))))
        if planes < od:
            run, fl = make(planes)
            return run, fl, f"batch item 0, {planes} of {od} output planes, all {d['Cout']} channels"
        # a whole batch item fits the budget: take as many items as it allows
        items = int(max(1, min(d["N"], target_s / max(dt * od / 2, 1e-3))))
        run, fl = make(od, items)
        return run, fl, f"batch items 0..{items - 1} of {d['N']}, all {od} output planes, all {d['Cout']} channels"

    def make(rows, items=1):
        xs = np.ascontiguousarray(t["x"][0:items, :, 0:rows])

        def run():
            t0 = time.perf_counter()
            oracle.dwsep_k(xs, t["w_dw"], t["w_pw"], t.get("b"))
            return time.perf_counter() - t0
        return run, 2.0 * items * rows * d["W"] * d["C"] * (d["K"] * d["K"] + d["Cout"])
    one, _ = make(8)
    dt = one()
    rows = int(max(8, min(d["H"], 8 * target_s / max(dt, 1e-3))))
    if rows < d["H"]:
        run, fl = make(rows)
        return run, fl, f"batch item 0, first {rows} of {d['H']} rows, all {d['Cout']} channels"
    items = int(max(1, min(d["N"], target_s / max(dt * d["H"] / 8, 1e-3))))
    run, fl = make(d["H"], items)
    return run, fl, f"batch items 0..{items - 1} of {d['N']}, all {d['H']} rows, all {d['Cout']} channels"


def cpu_baseline_sample(wl, target_s: float) -> dict:
    """Time the oracle, as it stands, on a bounded sample of the workload."""
    import oracle
    run, fl, sample = oracle_sample(wl, target_s)
    dt = run()
    return {"value": fl / dt / 1e9, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample, "seconds": dt}


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist_on = world > 1
    torch.cuda.set_device(local)
    if dist_on:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import implicit_gemm_convolution_x3x3_gb300 as ig3

    peaks, src = load_peaks()
    wl = WORKLOADS[args.workload]()
    sampler = ClockSampler(local) if rank == 0 else None
    res = measure_workload(ig3, wl, args.path, args.steps, args.warmup, peaks, src, rank, world, dist_on)
    clocks = sampler.summary(res["t0"], res["t1"]) if sampler else None

    e2e = None
    if rank == 0:
        e2e_k = max(3, min(args.steps, 20))
        ms, h2d, d2h = e2e_steps(ig3, wl, args.path, res["dev_t"], e2e_k, 3)
        link = host_link_peaks()
        step_s = ms * 1e-3 / e2e_k
        achieved = (h2d + d2h) / step_s / 1e9
        e2e = {"value": 2.0 * macs(wl) / step_s / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_k, "ms_per_step": 1e3 * step_s,
               "host_link": dict(link, achieved_gbs=round(achieved, 1),
                                 frac_of_concurrent=round(achieved / link["concurrent_gbs"], 3))}

    others = []
    if rank == 0 and not args.no_others and world == 1:
        for name in ["tiny", "conv3d_pool_reduce", "dwsep", "sweep16", "sweep64", "sweep128", "conv3d_same",
                     "conv3d_s2", "dwsep_k5"]:
            if name == args.workload:
                continue
            owl = WORKLOADS[name]()
            k = 200 if name == "tiny" else 10
            r = measure_workload(ig3, owl, "auto", k, 3, peaks, src)
            dev = device_us(r["call"], 50 if name == "tiny" else 5, 3)
            others.append({"workload": name, "desc": describe(owl), "path": r["path"],
                           "us_per_call": round(r["us_per_call"], 2), "gflops": round(r["gflops"], 1),
                           "device_us_per_call": None if dev is None else round(dev, 2),
                           "roofline": {k2: (round(v, 4) if isinstance(v, float) else v)
                                        for k2, v in r["roofline"].items()}})
            del r
            torch.cuda.empty_cache()
    if sampler:
        sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(wl, target_s=args.cpu_seconds)

    if rank != 0:
        if dist_on:
            dist.destroy_process_group()
        return
    rd, wr = compulsory_bytes(wl)
    roof = dict(res["roofline"])
    kernel_key = "conv3d_tc" if (res["path"] == "tc" and wl.op == "conv3d") else \
        ("conv3d_fma" if wl.op == "conv3d" else f"dwsep_{res['path']}")
    roof["traffic"] = traffic_for(kernel_key, wl.name)
    roof["algorithmic_per_launch"] = (2.0 * macs(wl) / 1e12 if roof["unit"] == "TFLOP/s" else (rd + wr) / 1e9)
    roof["algorithmic_unit"] = "TFLOP" if roof["unit"] == "TFLOP/s" else "GB"
    line = {
        "metric": METRIC, "value": res["gflops"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_total"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "impl": "ours",
        "data": "synthetic: seeded SplitMix64 draws, x ~ N(0,1), w and b ~ U(+-1/sqrt(27*Cin))",
        "config": {"workload": describe(wl), "name": wl.name, "global_batch": wl.dims["N"] * world,
                   "path": res["path"], "arith": ("3xTF32 on tcgen05 tensor cores, fp32 accumulate"
                                                  if res["path"] == "tc" else "fp32 FMA"),
                   "l2": (("inputs larger than L2" if rd > L2_BYTES else "working set NOT larger than L2 (no flush)")
                          + " (%.0f MB read, %.0f MB written per step; L2 %d MB)"
                          % (rd / 1e6, wr / 1e6, L2_BYTES // 2**20)),
                   "parallelism": f"batch shard per GPU x{world}" if world > 1 else "single GPU",
                   "us_per_call": res["us_per_call"]},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": res["timed_launches"],
        "clocks": clocks, "other_workloads": others,
    }
    print(json.dumps(line))
    if dist_on:
        dist.destroy_process_group()


def run_reference(args) -> None:
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    wl = WORKLOADS[args.workload]()
    # Size each step so the whole --warmup + --steps run stays within about two minutes.
    per_step = max(0.1, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    run, fl, sample = oracle_sample(wl, per_step)
    for _ in range(args.warmup):
        run()
    secs = sum(run() for _ in range(args.steps))
    value = fl * args.steps / secs / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic: seeded SplitMix64 draws (same inputs as the GPU arm)",
        "config": {"workload": describe(wl), "name": wl.name, "global_batch": wl.dims["N"],
                   "arith": "float64 nested loops (the oracle)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"each step: {sample}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_dwsep_crossover(args) -> None:
    """Depthwise-separable path study: both paths timed (CUDA events, inputs resident) over
    a grid of small images and channel counts; one JSON line per shape with the faster
    path and the one IG3_PATH_AUTO takes."""
    import torch
    import implicit_gemm_convolution_x3x3_gb300 as ig3
    torch.cuda.set_device(0)
    shapes = [(n, c, hw, hw, co) for (n, hw) in ((1, 32), (1, 64), (2, 128), (4, 256))
              for c in (16, 32, 64) for co in (16, 32, 64, 128)]
    for (N, C, H, W, Cout) in shapes:
        wl = si.dwsep_workload(f"dwsep_{N}x{C}x{H}x{W}_c{Cout}", N, C, H, W, Cout, seed=700 + C + Cout)
        t = {k: torch.from_numpy(v).cuda() for k, v in wl.generate_all().items()}
        row = {"study": "dwsep_crossover", "N": N, "C": C, "H": H, "W": W, "Cout": Cout,
               "gflop": 2.0 * macs(wl) / 1e9,
               "auto": ig3.dwsep_conv2d_select_path(N, C, H, W, Cout, "auto")}
        for path in ("tc", "fma"):
            try:
                ig3.dwsep_conv2d_select_path(N, C, H, W, Cout, path)
            except ig3.Ig3Error:
                row[path + "_us"] = None
                continue
            call, _, _ = make_call(ig3, wl, t, path)
            ms, _, _ = time_steps(call, args.steps, args.warmup, False)
            row[path + "_us"] = round(1e3 * ms / args.steps, 2)
        timed = [p for p in ("tc", "fma") if row[p + "_us"] is not None]
        row["faster"] = min(timed, key=lambda p: row[p + "_us"])
        print(json.dumps(row), flush=True)


def device_us(call, reps: int, warmup: int):
    """Device time per call: the calls captured in a CUDA graph and the replay timed with
    CUDA events (no host overhead); None if the calls cannot be captured."""
    import torch
    try:
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(reps):
                    call()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        g.replay()
        end.record()
        torch.cuda.synchronize()
        return 1e3 * start.elapsed_time(end) / reps
    except Exception:  # noqa: BLE001  (capture unsupported: report host-inclusive times only)
        torch.cuda.synchronize()
        return None


def run_conv3d_crossover(args) -> None:
    """conv3d path study: both paths timed over small and medium shapes (Cin = Cout in
    16, 32, 64; tanh(mish)), plus the pool-reduce and 16-channel sweep workloads; one JSON
    line per shape with each path's device time (CUDA graph of the calls) and per-call
    time with host overhead (CUDA events around a loop of calls), the faster path and the
    one IG3_PATH_AUTO takes."""
    import torch
    import implicit_gemm_convolution_x3x3_gb300 as ig3
    torch.cuda.set_device(0)
    shapes = [(n, c, d, h, w, c, "tanh_mish") for n in (1, 4) for c in (16, 32, 64)
              for (d, h, w) in ((8, 16, 16), (8, 32, 32), (16, 32, 64), (16, 64, 64))]
    shapes += [(1, c, d, h, w, 16, "tanh_mish") for c in (1, 4, 8)
               for (d, h, w) in ((3, 3, 4), (4, 6, 8), (6, 10, 16), (8, 16, 32))]
    shapes += [(2, 4, 8, 8, 8, 16, "tanh_mish"), (2, 4, 8, 8, 8, 32, "tanh_mish"),
               (1, 8, 5, 7, 9, 48, "tanh_mish"), (1, 16, 6, 12, 20, 96, "tanh_mish")]
    shapes += [(128, 8, 16, 64, 64, 16, "pool_reduce"), (8, 16, 32, 64, 64, 16, "tanh_mish")]
    for (N, Cin, D, H, W, Cout, epi) in shapes:
        wl = si.conv3d_workload(f"conv3d_{N}x{Cin}x{D}x{H}x{W}_c{Cout}", N, Cin, D, H, W, Cout,
                                seed=800 + Cin + D + W, epilogue=epi, bias2=(epi == "pool_reduce"))
        t = {k: torch.from_numpy(v).cuda() for k, v in wl.generate_all().items()}
        row = {"study": "conv3d_crossover", "N": N, "Cin": Cin, "D": D, "H": H, "W": W, "Cout": Cout,
               "epilogue": epi, "gflop": 2.0 * macs(wl) / 1e9,
               "auto": ig3.conv3d_fused_select_path(N, Cin, D, H, W, Cout, epi, "auto")}
        reps = max(3, min(50, int(2e3 / max(row["gflop"], 1e-3) ** 0.5)))
        for path in ("tc", "fma"):
            try:
                ig3.conv3d_fused_select_path(N, Cin, D, H, W, Cout, epi, path)
            except ig3.Ig3Error:
                row[path + "_us"] = row[path + "_dev_us"] = None
                continue
            call, _, _ = make_call(ig3, wl, t, path)
            ms, _, _ = time_steps(call, reps, args.warmup, False)
            row[path + "_us"] = round(1e3 * ms / reps, 2)
            dev = device_us(call, reps, args.warmup)
            row[path + "_dev_us"] = None if dev is None else round(dev, 2)
            if ig3.ig3_last_device_status() != 0:
                raise RuntimeError("a kernel reported a device-side timeout during the study")
        timed = [p for p in ("tc", "fma") if row[p + "_us"] is not None]
        key = "_dev_us" if all(row[p + "_dev_us"] is not None for p in timed) else "_us"
        row["faster"] = min(timed, key=lambda p: row[p + key])
        print(json.dumps(row), flush=True)
        del t
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="conv3d_tanh_mish")
    ap.add_argument("--path", choices=["auto", "tc", "fma"], default="auto")
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads' summary")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample size in seconds")
    ap.add_argument("--study", choices=["dwsep_crossover", "conv3d_crossover"], default=None,
                    help="run a path study instead of the benchmark (JSON line per shape)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (smaller cases for profiling; not a bench line)")
    args = ap.parse_args()
    if args.batch > 0:
        base = WORKLOADS[args.workload]
        WORKLOADS[args.workload] = lambda: with_batch(base(), args.batch)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.study == "dwsep_crossover":
        run_dwsep_crossover(args)
    elif args.study == "conv3d_crossover":
        run_conv3d_crossover(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
