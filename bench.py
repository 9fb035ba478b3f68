#!/usr/bin/env python
"""Benchmark of the NA3D forward pass on GB300 (one JSON line on stdout).

A step is one na3d_fwd call over the whole workload: bf16 (B,T,H,W,NH,HD)
q, k, v resident in HBM, output written to HBM. The headline workload is the
largest benchmark shape, B=2, T=16, H=96, W=128, NH=16, HD=128 with a (3,7,7)
window; every benchmark shape (the headline included) is reported under
"configs", each on the seeded input recipe that the parity tests use.

Metric: useful TFLOPS = 4*B*T*H*W*NH*HD*KT*KH*KW / kernel time, and its
fraction of the GB300 roofline, where the roofline time is the slower of the
dense-bf16 tensor peak and the four tensors' bf16 bytes at HBM bandwidth
(measured peaks from MEASURED_PEAKS.json).

Timing: CUDA events on the launching stream around each kernel, L2 flushed
(a buffer of twice the L2 size is overwritten) between timed steps, a
barrier and a device synchronize on both sides of the K timed steps, and the
maximum over ranks. SM clocks are sampled with nvidia-smi during the timed
steps.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload: the deliberately slow baseline.

Multi-GPU (torchrun): every rank runs its own replica of the workload on its
own GPU; the path has no cross-GPU exchange ("scaling": "weak").
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
sys.path.insert(0, ROOT)

METRIC = "NA3D fwd useful TFLOPS and % of GB300 bf16 tensor roofline per config"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOADS = {
    # name: ((B, T, H, W, NH, HD), (KT, KH, KW))
    "na3d_b1_t4_h8_w16_nh2_hd32_k3x5x5": ((1, 4, 8, 16, 2, 32), (3, 5, 5)),
    "na3d_b1_t16_h64_w64_nh8_hd64_k3x7x7": ((1, 16, 64, 64, 8, 64), (3, 7, 7)),
    "na3d_b1_t16_h64_w96_nh8_hd64_k3x5x5": ((1, 16, 64, 96, 8, 64), (3, 5, 5)),
    "na3d_b1_t16_h64_w5_nh8_hd64_k3x5x5": ((1, 16, 64, 5, 8, 64), (3, 5, 5)),
    "na3d_b1_t16_h48_w48_nh8_hd64_k11x11x11": ((1, 16, 48, 48, 8, 64), (11, 11, 11)),
    "na3d_b2_t16_h96_w128_nh16_hd128_k3x7x7": ((2, 16, 96, 128, 16, 128), (3, 7, 7)),
    "na3d_b2_t8_h64_w33_nh8_hd64_k3x7x33": ((2, 8, 64, 33, 8, 64), (3, 7, 33)),
}
HEADLINE = "na3d_b2_t16_h96_w128_nh16_hd128_k3x7x7"
# Smaller cases of the same kernel instances for ncu captures (inputs still
# larger than L2); selectable with --workload, not part of the configs table.
PROFILE_WORKLOADS = {
    "na3d_b1_t16_h48_w64_nh16_hd128_k3x7x7": ((1, 16, 48, 64, 16, 128), (3, 7, 7)),
}
ALL_WORKLOADS = {**WORKLOADS, **PROFILE_WORKLOADS}


def useful_flops(shape, kernel):
    B, T, H, W, NH, HD = shape
    return 4.0 * B * T * H * W * NH * HD * kernel[0] * kernel[1] * kernel[2]


def min_bytes(shape):
    n = 1
    for d in shape:
        n *= d
    return 4.0 * n * 2  # q, k, v read once, out written once, bf16


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# NVIDIA's published dense (no sparsity) bf16 tensor throughput of one GB300
# GPU, for context beside the measured peaks
NOMINAL_BF16_TFLOPS = 2250.0


def roofline_terms(shape, kernel, seconds, peaks, tc_tflops=None):
    flops, nbytes = useful_flops(shape, kernel), min_bytes(shape)
    t_tc = flops / ((tc_tflops or peaks["bf16_tflops"]) * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    return {
        "bound": bound,
        "useful_tflops": flops / seconds / 1e12,
        "roofline_frac": max(t_tc, t_hbm) / seconds,
        "achieved_gbs": nbytes / seconds / 1e9,
        "roofline_us": max(t_tc, t_hbm) * 1e6,
    }


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "neighborhood_attention_video_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_sha") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "clocks.mem,clocks.max.mem")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summarize(self.lines)

    @classmethod
    def summarize(cls, lines):
        """Median SM and memory clocks, maximum clocks, median power and the
        throttle reasons seen active, from `nvidia-smi --query-gpu=FIELDS
        --format=csv,noheader,nounits` lines."""
        sm, smax, mem, mmax, power, reasons = [], [], [], [], [], set()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(cls.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
            for dst, i in ((power, 3), (mem, 9), (mmax, 10)):
                try:
                    dst.append(float(parts[i]))
                except (ValueError, IndexError):
                    pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "mem_max_mhz": max(mmax) if mmax else None,
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
        pg = dist
    if args.impl == "ours":
        torch.cuda.set_device(local)
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def allreduce_max(pg, x):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def gpu_uuid(local):
    import torch
    try:
        u = torch.cuda.get_device_properties(local).uuid
        return f"GPU-{u}"
    except Exception:
        return local


def time_kernel(shape, kernel, q, k, v, out, steps, warmup, flush, stream):
    """Per-step CUDA-event kernel times (s) with the L2 flushed between steps
    (flush None: back to back, inputs left in L2 by the previous step)."""
    import torch
    import neighborhood_attention_video_gb300 as na
    for _ in range(warmup):
        na.na3d_fwd(q, k, v, out, kernel, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            na.na3d_fwd(q, k, v, out, kernel, stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e-3 for a, b in evs]


def run_ours(args):
    import numpy as np
    import torch

    import na3d_inputs
    import neighborhood_attention_video_gb300 as na

    world, rank, local, pg = dist_setup(args)
    peaks, peak_src = load_peaks()
    shape, kernel = ALL_WORKLOADS[args.workload]
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    # inputs: the seeded recipe, generated into pinned host memory, then resident in HBM
    n = int(np.prod(shape))
    host = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    na3d_inputs.fill_qkv_host(*(t.data_ptr() for t in host), shape, seed=args.seed)
    q, k, v = (t.to(dev) for t in host)
    out = torch.empty_like(q)
    host_out = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    # warm-up, then K timed steps bracketed by barrier + synchronize
    for _ in range(args.warmup):
        na.na3d_fwd(q, k, v, out, kernel, stream=stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_uuid(local))
    clocks.start()
    barrier(pg)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    per_step = time_kernel(shape, kernel, q, k, v, out, args.steps, 0, flush, stream)
    torch.cuda.synchronize()
    barrier(pg)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    kernel_s = allreduce_max(pg, sum(per_step)) / args.steps
    status = na.na3d_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status}: {na.na3d_status_string(status)}")

    flops = useful_flops(shape, kernel)
    terms = roofline_terms(shape, kernel, kernel_s, peaks)
    value = world * flops / kernel_s / 1e12
    plan = na.na3d_plan(*shape[1:], *kernel)
    executed = executed_flops(shape, plan)

    # e2e: every step copies its q, k, v from pinned host memory to HBM, runs the kernel and
    # copies its output back to pinned host memory. Steps are pipelined as a serving loop runs
    # them: two device buffer sets, the copy-in of step i+1 and the copy-out of step i-1 on
    # their own streams while step i computes; a buffer set is refilled only after the step
    # that used it has finished with it.
    e2e_steps = max(3, min(args.steps, 30))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs = [(q, k, v, out), tuple(torch.empty_like(q) for _ in range(4))]
    host_outs = [host_out, torch.empty(shape, dtype=torch.bfloat16).pin_memory()]

    def pipeline(steps):
        """`steps` pipelined steps; returns the device time from the first
        copy-in to the last copy-out (s)."""
        done_compute, done_out = [None, None], [None, None]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(pg)
        start.record(s_in)
        for i in range(steps):
            j = i % 2
            qb, kb, vb, ob = bufs[j]
            with torch.cuda.stream(s_in):
                if done_compute[j] is not None:
                    s_in.wait_event(done_compute[j])
                for dst, src in zip((qb, kb, vb), host):
                    dst.copy_(src, non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(s_in)
            stream.wait_event(copied)
            if done_out[j] is not None:
                stream.wait_event(done_out[j])
            na.na3d_fwd(qb, kb, vb, ob, kernel, stream=stream)
            done_compute[j] = torch.cuda.Event()
            done_compute[j].record(stream)
            s_out.wait_event(done_compute[j])
            with torch.cuda.stream(s_out):
                host_outs[j].copy_(ob, non_blocking=True)
                done_out[j] = torch.cuda.Event()
                done_out[j].record(s_out)
        end.record(s_out)   # after the last copy-out, which follows every earlier step's work
        torch.cuda.synchronize()
        barrier(pg)
        return start.elapsed_time(end) * 1e-3

    pipeline(max(3, args.warmup // 4))   # untimed: first use of the buffers, streams and pinned pages
    e2e_s = allreduce_max(pg, pipeline(e2e_steps)) / e2e_steps
    _ = float(host_out.view(torch.int16)[0, 0, 0, 0, 0, 0].item())  # the read-back result

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": kernel_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: q,k,v iid N(0,1) rounded to bf16, q pre-scaled by HD^-0.5, seed %d" % args.seed,
        "config": {
            "workload": args.workload,
            "shape_BTHWNH_HD": list(shape),
            "kernel": list(kernel),
            "l2": "flushed between timed steps (2x L2 buffer overwritten)",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "plan": {k2: plan[k2] for k2 in ("bt", "bh", "bw", "cw", "cr", "n_mma", "tile_cap", "w_stride")},
        },
        "roofline": {
            "bound": terms["bound"],
            "achieved": terms["achieved_gbs"] if terms["bound"] == "hbm" else terms["useful_tflops"],
            "peak": peaks["hbm_gbs"] if terms["bound"] == "hbm" else peaks["bf16_tflops"],
            "unit": "GB/s" if terms["bound"] == "hbm" else "TFLOP/s",
            "frac": terms["roofline_frac"],
            "peak_source": peak_src,
            "traffic": ncu_traffic(args.workload),
            "algorithmic_bytes": min_bytes(shape),
            "useful_flops": flops,
            "executed_mma_flops": executed,
            "executed_tflops": executed / kernel_s / 1e12,
            "kernel_us": kernel_s * 1e6,
            "roofline_us": terms["roofline_us"],
        },
        "e2e": {
            "value": world * flops / e2e_s / 1e12,
            "unit": "TFLOPS",
            "h2d_bytes_per_step": 3 * n * 2,
            "d2h_bytes_per_step": n * 2,
            "ms_per_step": e2e_s * 1e3,
            "steps": e2e_steps,
            "mode": "steps pipelined over two device buffer sets: copy-in, kernel and copy-out "
                    "on separate streams",
        },
        "gpu_launches": args.steps,
        "clocks": clk,
        "timed_wall_s": wall,
    }

    if rank == 0 and not args.no_configs:
        result["configs"] = per_config_table(dev, stream, flush, peaks,
                                             resident={args.workload: (q, k, v, out)}
                                             if args.seed == 0 else None)
        result["qkv_projection"] = projection_line(shape, dev, stream, flush, peaks)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(shape, kernel, args.seed, budget_s=args.cpu_seconds)
        if not args.no_configs:
            result["cpu_oracle_per_config"] = cpu_per_config(args.seed)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def seeded_inputs(shape, dev, seed=0):
    """q, k, v of the seeded recipe (the parity tests' inputs), generated in
    pinned host memory and copied to the device."""
    import torch
    import na3d_inputs
    host = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    na3d_inputs.fill_qkv_host(*(t.data_ptr() for t in host), shape, seed=seed)
    return [t.to(dev) for t in host]


def per_config_table(dev, stream, flush, peaks, resident=None, steps=20, warmup=3):
    """Every benchmark shape: useful TFLOPS and roofline fraction, on the
    seeded input recipe (seed 0). `resident` maps a workload name to its
    (q, k, v, out) already on the device. A row whose launches report a
    pipeline wait that ran out raises instead of being recorded."""
    import torch
    import neighborhood_attention_video_gb300 as na
    table = {}
    resident = resident or {}
    for name, (shape, kernel) in WORKLOADS.items():
        if name in resident:
            q, k, v, out = resident[name]
        else:
            q, k, v = seeded_inputs(shape, dev)
            out = torch.empty_like(q)
        times = time_kernel(shape, kernel, q, k, v, out, steps, warmup, flush, stream)
        t = statistics.median(times)
        t_warm = statistics.median(time_kernel(shape, kernel, q, k, v, out, steps, 1, None, stream))
        status = na.na3d_device_status(stream)
        if status != 0:
            raise RuntimeError(f"{name}: device status {status}: {na.na3d_status_string(status)}")
        terms = roofline_terms(shape, kernel, t, peaks)
        sustained = roofline_terms(shape, kernel, t, peaks, peaks["bf16_tflops_sustained"])
        nominal = roofline_terms(shape, kernel, t, peaks, NOMINAL_BF16_TFLOPS)
        plan = na.na3d_plan(*shape[1:], *kernel)
        executed = executed_flops(shape, plan)
        table[name] = {
            "us": t * 1e6,
            "useful_tflops": terms["useful_tflops"],
            "roofline_frac": terms["roofline_frac"],
            "bound": terms["bound"],
            "roofline_us": terms["roofline_us"],
            "roofline_frac_sustained_tc": sustained["roofline_frac"],
            "roofline_frac_nominal_tc": nominal["roofline_frac"],
            "us_warm": t_warm * 1e6,
            "executed_tflops": executed / t / 1e12,
            "executed_over_useful": executed / useful_flops(shape, kernel),
            # brick bt x bh x bw, chunk rows cr of cw keys, tile width n_mma, tile cap, W row stride
            "plan": [plan["bt"], plan["bh"], plan["bw"], plan["cw"], plan["cr"], plan["n_mma"],
                     plan["tile_cap"], plan["w_stride"]],
            "traffic": ncu_traffic(name),
            "inputs": "seeded recipe, seed 0",
        }
        if name not in resident:
            del q, k, v, out
    torch.cuda.synchronize()
    return table


def executed_flops(shape, plan):
    """MMA flops the plan issues: every chunk is a 128-row score tile of
    n_mma columns and its product, each 2 * HD flops per element."""
    return plan["chunks_per_slice"] * shape[0] * shape[4] * 128 * plan["n_mma"] * shape[5] * 4.0


def projection_line(shape, dev, stream, flush, peaks, steps=20, warmup=3):
    """The fused QKV projection that produces this workload's q, k, v:
    x (B*T*H*W tokens, C = NH*HD channels) times a (3*NH*HD, C) weight with
    a bias; a dense contraction, so its roofline is the bf16 tensor peak."""
    import torch
    import neighborhood_attention_video_gb300 as na
    B, T, H, W, NH, HD = shape
    M, C, N = B * T * H * W, NH * HD, 3 * NH * HD
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    x = torch.randn((M, C), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((N, C), generator=gen, device=dev, dtype=torch.float32) / math.sqrt(C)).to(torch.bfloat16)
    bias = torch.randn((N,), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    qkv = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for _ in range(warmup):
        na.na3d_qkv_proj(x, w, bias, qkv, NH, HD, stream=stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            na.na3d_qkv_proj(x, w, bias, qkv, NH, HD, stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    status = na.na3d_device_status(stream)
    if status != 0:
        raise RuntimeError(f"qkv projection: device status {status}: {na.na3d_status_string(status)}")
    t = statistics.median(a.elapsed_time(b) * 1e-3 for a, b in evs)
    flops = 2.0 * M * C * N
    nbytes = 2.0 * (M * C + N * C + M * N)
    del x, w, bias, qkv
    return {
        "shape_M_C_N": [M, C, N], "us": t * 1e6, "tflops": flops / t / 1e12,
        "frac_of_bf16_peak": flops / t / 1e12 / peaks["bf16_tflops"],
        "hbm_gbs": nbytes / t / 1e9,
        "roofline_us": max(flops / (peaks["bf16_tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9)) * 1e6,
    }


# ---------------------------------------------------------------- CPU oracle

def oracle_sample_rate(shape, kernel, seed, budget_s, nthreads):
    """Time the fp64 oracle on a random sample of output rows of the workload,
    sized to take about `budget_s`; returns (useful TFLOPS, rows, seconds)."""
    import numpy as np

    import na3d_inputs
    import oracle
    q, k, v = na3d_inputs.make_qkv(*shape, seed=seed)
    total = int(np.prod(shape[:5]))
    per_row = 4.0 * shape[5] * kernel[0] * kernel[1] * kernel[2]
    rng = np.random.default_rng(seed)
    # grow the sample until it takes at least half the budget (a small probe
    # is dominated by fixed costs) or covers the whole workload
    n = min(total, 2048)
    for _ in range(5):
        rows = rng.choice(total, size=n, replace=False)
        t0 = time.perf_counter()
        oracle.na3d_fwd_rows(q, k, v, kernel, rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * budget_s or n == total:
            break
        n = int(min(total, max(2 * n, 0.9 * n * budget_s / max(dt, 1e-6))))
    return per_row * n / dt / 1e12, n, dt


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        txt = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in txt.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(shape, kernel, seed, budget_s=10.0):
    cores = os.cpu_count() or 1
    tf, n, dt = oracle_sample_rate(shape, kernel, seed, budget_s, cores)
    return {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "machine": os.uname().machine,
            "sample": f"{n} random output rows (b,t,h,w,head) of the workload, fp64 oracle, {dt:.1f} s"}


# configurations whose oracle is also timed on one thread
SINGLE_THREAD_CONFIGS = ("na3d_b1_t4_h8_w16_nh2_hd32_k3x5x5", "na3d_b1_t16_h64_w5_nh8_hd64_k3x5x5",
                         "na3d_b2_t8_h64_w33_nh8_hd64_k3x7x33")


def cpu_per_config(seed, budget_s=1.5):
    """The fp64 oracle's useful GFLOP/s for every benchmark configuration, on
    all host cores (and on one thread for the small ones). A row's work
    depends only on the head dim and the window, so each is timed on rows of
    a grid cut to at most 2K + 8 per axis and two heads (same HD, window and
    border mix), which keeps input generation short."""
    cores = os.cpu_count() or 1
    table = {}
    for name, (shape, kernel) in WORKLOADS.items():
        B, T, H, W, NH, HD = shape
        small = (1, min(T, 2 * kernel[0] + 8), min(H, 2 * kernel[1] + 8), min(W, 2 * kernel[2] + 8),
                 min(NH, 2), HD)
        tf, n, dt = oracle_sample_rate(small, kernel, seed, budget_s, cores)
        row = {"gflops_all_cores": tf * 1e3, "cores": cores, "rows": n, "grid": list(small)}
        if name in SINGLE_THREAD_CONFIGS:
            tf1, n1, _ = oracle_sample_rate(small, kernel, seed, budget_s, 1)
            row["gflops_1_thread"] = tf1 * 1e3
        table[name] = row
    return table


# The pages' own kernel benchmark shapes ("[Triton/Gluon] Add 3D neighborhood
# flash attention (na3d_flash)", review thread, Performance table): B = 1,
# HD = 64, with the gfx950 (MI350X) times of the Triton kernel, which include
# a staging copy of v. The pages leave NH open (4, 8 or 32); NH = 8 here.
PAGES_SHAPES = [
    ((1, 18, 32, 48, 8, 64), (3, 7, 7), 1249.0),
    ((1, 36, 64, 96, 8, 64), (3, 5, 5), 1910.0),
    ((1, 40, 96, 96, 8, 64), (3, 5, 5), 3319.0),
    ((1, 16, 80, 32, 8, 64), (11, 11, 11), 1153.0),
    ((1, 79, 192, 192, 8, 64), (11, 11, 11), 99143.0),
    ((1, 4, 8, 128, 8, 64), (3, 5, 27), 40.0),
]


def run_pages_shapes(args):
    """Times the kernel on the pages' benchmark shapes (context: another
    vendor's GPU and an unstated NH), L2 flushed between steps."""
    import torch
    import neighborhood_attention_video_gb300 as na
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    peaks, _ = load_peaks()
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024,
                        dtype=torch.float32, device=dev)
    rows = []
    gen = torch.Generator(device=dev)
    for shape, kernel, gfx950_us in PAGES_SHAPES:
        gen.manual_seed(args.seed)
        q = (torch.randn(shape, generator=gen, device=dev) * shape[-1] ** -0.5).to(torch.bfloat16)
        k = torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        t = statistics.median(time_kernel(shape, kernel, q, k, v, out, 20, 3, flush, stream))
        terms = roofline_terms(shape, kernel, t, peaks)
        rows.append({"shape_BTHWNH_HD": list(shape), "kernel": list(kernel), "us": t * 1e6,
                     "useful_tflops": terms["useful_tflops"], "roofline_frac": terms["roofline_frac"],
                     "pages_gfx950_us": gfx950_us})
        del q, k, v, out
    print(json.dumps({"pages_shapes": rows, "note": "NH = 8 assumed; the pages' times are for "
                      "AMD MI350X and include a staging copy of v"}), flush=True)


def run_proj_only(args):
    """The fused QKV projection of the workload alone (one line; the command
    the projection's ncu capture runs)."""
    import torch
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    peaks, _ = load_peaks()
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size // 4 + 1024,
                        dtype=torch.float32, device=dev)
    shape, _ = ALL_WORKLOADS[args.workload]
    line = projection_line(shape, dev, stream, flush, peaks, steps=args.steps, warmup=args.warmup)
    print(json.dumps({"qkv_projection": line, "workload": args.workload}), flush=True)


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return
    import numpy as np

    import na3d_inputs
    import oracle
    shape, kernel = ALL_WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    q, k, v = na3d_inputs.make_qkv(*shape, seed=args.seed)
    total = int(np.prod(shape[:5]))
    per_row = 4.0 * shape[5] * kernel[0] * kernel[1] * kernel[2]
    rng = np.random.default_rng(args.seed)
    # size each step so the whole run stays within about args.cpu_seconds * 6
    probe = rng.choice(total, size=min(total, 512), replace=False)
    t0 = time.perf_counter()
    oracle.na3d_fwd_rows(q, k, v, kernel, probe, nthreads=cores)
    rate = probe.size / max(time.perf_counter() - t0, 1e-6)
    budget = 6.0 * args.cpu_seconds
    rows_per_step = int(max(64, min(total, rate * budget / (args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle.na3d_fwd_rows(q, k, v, kernel, rng.choice(total, size=rows_per_step), nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.na3d_fwd_rows(q, k, v, kernel, rng.choice(total, size=rows_per_step), nthreads=cores)
    dt = time.perf_counter() - t0
    value = per_row * rows_per_step * args.steps / dt / 1e12
    res = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same recipe and seed)",
        "config": {"workload": args.workload, "shape_BTHWNH_HD": list(shape), "kernel": list(kernel)},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} random output rows per step"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(res), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(ALL_WORKLOADS), default=HEADLINE)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pages-shapes", action="store_true",
                    help="time the pages' own benchmark shapes (context) and exit")
    ap.add_argument("--proj-only", action="store_true",
                    help="time only the fused QKV projection of --workload and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.pages_shapes:
        run_pages_shapes(args)
    elif args.proj_only:
        run_proj_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
