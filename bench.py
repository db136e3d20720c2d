#!/usr/bin/env python3
"""Benchmark of the W4A16 decode path on GB300 -- prints ONE JSON line.

Headline step: one pass of the Llama-3-8B decode linear layers at M = 1
(QKV 6144x4096, O 4096x4096, gate/up 28672x4096, down 4096x14336, lm_head
128256x4096) through ``w4a16_gemm``, weights already resident in HBM in the
kernel layout.  The step moves 383.7 MB of packed weights and scales -- three
times the 129 MB L2 -- so every step streams from HBM (no L2 flush needed).
``value`` is algorithmic bytes / device time (GB/s): bytes per call =
N*K/2 + 2*N*K/128 + 2*M*K + 2*M*N.

Also reported in the same line: per-shape us/call over rotating weight copies
(>= 4x L2), the 8B-stack token (129 GEMVs, tokens/s), the M = 2..16 sweep over
the Llama and Qwen-2.5-7B shapes, the quantizer on [14336, 4096], the
roofline of the GEMV kernel, the CPU oracle baseline on the host cores, the
end-to-end number through the Python API with host buffers, and SM clocks
sampled during the timed region.

``--impl reference`` times the CPU oracle (the only reference this path has)
on the same workload, a bounded sample of rows per step.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from w4a16_weight_only_gemm_gb300 import synthetic, workloads  # noqa: E402

METRIC = "W4A16 GEMV achieved HBM GB/s (% of 8 TB/s) and 8B-stack tokens/s at M=1"
WORKLOAD = ("llama3_8b_decode_m1: qkv 6144x4096, o_proj 4096x4096, gate_up 28672x4096, "
            "down 4096x14336, lm_head 128256x4096; M=1; W4A16 group 128, fp16 scales")
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--skip-extras", action="store_true",
                   help="headline step only (no per-shape, stack, sweep, quantizer sections)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="budget of the CPU oracle baseline sample")
    p.add_argument("--section", choices=("prefill", "quantizer", "stack", "per_shape", "formats",
                                         "formats_prefill"),
                   default=None,
                   help="run one section alone and print its JSON (profiling aid; not the "
                        "benchmark line)")
    return p.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs the same step on its GPU)
# ----------------------------------------------------------------------------
def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                cols = [c.strip() for c in line.split(",")]
                if len(cols) < 9:
                    continue
                try:
                    sm.append(float(cols[1]))
                    smax.append(float(cols[2]))
                    power.append(float(cols[3]))
                except ValueError:
                    continue
                for name, val in zip(names, cols[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# GPU side
# ----------------------------------------------------------------------------
PARITY_ROWS = 64  # sampled rows of every timed layer checked against the oracle
STEPS_PER_GRAPH = 10  # headline steps captured per CUDA graph replay


def make_layer(lin, workload: str, idx: int, M: int = 1, keep_rows: int = 0):
    """A quantized layer on the GPU; with keep_rows, the master weight's rows
    at `keep_rows` sampled indices are kept on the host (the oracle quantizes
    them itself for the parity check of the CPU-baseline leg)."""
    import w4a16_weight_only_gemm_gb300 as w4
    sw, sx = synthetic.seeds(workload, idx)
    W = synthetic.master_weight(lin.N, lin.K, sw, device="cuda")
    q, s = w4.quantize(W)
    r = w4.repack(q)
    layer = {"lin": lin, "r": r, "s": s, "M": M}
    if keep_rows:
        rows = np.sort(np.random.default_rng(sw).choice(lin.N, size=min(keep_rows, lin.N),
                                                        replace=False))
        layer["rows"] = rows
        layer["W_rows"] = W[torch.from_numpy(rows).cuda()].cpu()
    del W, q
    layer["x"] = synthetic.activations(M, lin.K, sx, device="cuda")
    layer["y"] = torch.empty((M, lin.N), dtype=torch.float16, device="cuda")
    return layer


def gemm_call(layer, r=None, s=None):
    import w4a16_weight_only_gemm_gb300 as w4
    w4.gemm(layer["x"], layer["r"] if r is None else r, layer["s"] if s is None else s,
            out=layer["y"])


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # first use outside capture: per-device set-up
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, stream, reps: int, warmup: int, world: int = 1) -> float:
    """Seconds per replay (CUDA events on the replay stream, max over ranks)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    secs = start.elapsed_time(end) / 1e3
    return max_over_ranks(secs, world) / reps


def l2_bytes() -> int:
    try:
        return int(torch.cuda.get_device_properties(0).L2_cache_size)
    except AttributeError:
        return 129 * 2 ** 20


def per_shape_us(lin, workload, idx, M=1, reps=20):
    """us per call over rotating weight copies totalling >= 4x L2."""
    base = make_layer(lin, workload, idx, M)
    nbytes = lin.N * lin.K // 2 + 2 * lin.N * (lin.K // 128)
    copies = max(2, -(-4 * l2_bytes() // nbytes))
    rs = [base["r"]] + [base["r"].clone() for _ in range(copies - 1)]
    ss = [base["s"]] + [base["s"].clone() for _ in range(copies - 1)]
    stream = torch.cuda.Stream()

    def body():
        for r, s in zip(rs, ss):
            gemm_call(base, r, s)
    g = capture(body, stream)
    t = time_graph(g, stream, reps, 3) / copies
    b = workloads.algorithmic_bytes(M, lin.N, lin.K)
    del rs, ss, g
    return {"us": round(t * 1e6, 3), "gbs": round(b / t / 1e9, 1), "bytes": b, "copies": copies}


def formats_m1():
    """The format variants (w4a16_gemm_ex) on the Llama-3-8B decode shapes at
    M = 1: us per call over rotating weight copies (>= 4x L2), GB/s of the
    variant's algorithmic bytes (its scales and zero points included)."""
    import w4a16_weight_only_gemm_gb300 as w4
    out = {}
    formats = [(32, False), (32, True), (64, False), (128, True), (w4.PER_CHANNEL, False),
               (w4.PER_CHANNEL, True), (128, "awq")]
    stream = torch.cuda.Stream()
    for group, asym in formats:
        awq = asym == "awq"  # group 128 symmetric codes with an AWQ activation scale
        asym = False if awq else asym
        name = ("g" + str(group) if group > 0 else "per_channel") + ("_asym" if asym else "_sym")
        name += "_awq" if awq else ""
        res = {}
        for i, lin in enumerate(workloads.LLAMA3_8B):
            sw, sx = synthetic.seeds("llama3_8b_decode", i)
            W = synthetic.master_weight(lin.N, lin.K, sw, device="cuda")
            q, s, z = w4.quantize_ex(W, group, asymmetric=asym)
            r = w4.repack(q)
            del W, q
            x = synthetic.activations(1, lin.K, sx, device="cuda")
            alpha = (torch.rand(lin.K, device="cuda") * 1.5 + 0.5).half() if awq else None
            y = torch.empty((1, lin.N), dtype=torch.float16, device="cuda")
            nbytes = r.numel() + s.numel() * 2 + (z.numel() if z is not None else 0)
            copies = max(2, -(-4 * l2_bytes() // nbytes))
            rs = [r] + [r.clone() for _ in range(copies - 1)]

            def body():
                for rr in rs:
                    w4.gemm_ex(x, rr, s, z, group, out=y, alpha=alpha)
            g = capture(body, stream)
            t = time_graph(g, stream, 10, 3) / copies
            b = workloads.algorithmic_bytes(1, lin.N, lin.K, group, asym) + (2 * lin.K if awq else 0)
            res[lin.name] = {"us": round(t * 1e6, 3), "gbs": round(b / t / 1e9, 1)}
            del rs, g, r, s, z
        tot_t = sum(v["us"] for v in res.values())
        tot_b = sum(workloads.algorithmic_bytes(1, l.N, l.K, group, asym) + (2 * l.K if awq else 0)
                    for l in workloads.LLAMA3_8B)
        res["five_shapes"] = {"us": round(tot_t, 2), "gbs": round(tot_b / tot_t / 1e3, 1)}
        out[name] = res
        torch.cuda.empty_cache()
    # W8A16 (per-channel INT8): codes [N, K] bytes + fp16 scale per row
    res = {}
    for i, lin in enumerate(workloads.LLAMA3_8B):
        sw, sx = synthetic.seeds("llama3_8b_decode", i)
        W = synthetic.master_weight(lin.N, lin.K, sw, device="cuda")
        q, s = w4.quantize_w8(W)
        del W
        x = synthetic.activations(1, lin.K, sx, device="cuda")
        y = torch.empty((1, lin.N), dtype=torch.float16, device="cuda")
        copies = max(2, -(-4 * l2_bytes() // q.numel()))
        qs = [q] + [q.clone() for _ in range(copies - 1)]

        def body():
            for qq in qs:
                w4.gemm_w8(x, qq, s, out=y)
        g = capture(body, stream)
        t = time_graph(g, stream, 10, 3) / copies
        b = lin.N * lin.K + 2 * lin.N + 2 * lin.K + 2 * lin.N
        res[lin.name] = {"us": round(t * 1e6, 3), "gbs": round(b / t / 1e9, 1)}
        del qs, g, q, s
    tot_t = sum(v["us"] for v in res.values())
    tot_b = sum(l.N * l.K + 4 * l.N + 2 * l.K for l in workloads.LLAMA3_8B)
    res["five_shapes"] = {"us": round(tot_t, 2), "gbs": round(tot_b / tot_t / 1e3, 1)}
    out["w8a16_per_channel"] = res
    torch.cuda.empty_cache()
    # GGUF Q4_0 blocks: 18 bytes per 32 weights (scales inline)
    res = {}
    for i, lin in enumerate(workloads.LLAMA3_8B):
        sw, sx = synthetic.seeds("llama3_8b_decode", i)
        W = synthetic.master_weight(lin.N, lin.K, sw, device="cuda")
        blk = w4.quantize_q4_0(W)
        del W
        x = synthetic.activations(1, lin.K, sx, device="cuda")
        y = torch.empty((1, lin.N), dtype=torch.float16, device="cuda")
        copies = max(2, -(-4 * l2_bytes() // blk.numel()))
        bs = [blk] + [blk.clone() for _ in range(copies - 1)]

        def body():
            for bb in bs:
                w4.gemm_q4_0(x, bb, out=y)
        g = capture(body, stream)
        t = time_graph(g, stream, 10, 3) / copies
        b = lin.N * lin.K // 32 * 18 + 2 * lin.K + 2 * lin.N
        res[lin.name] = {"us": round(t * 1e6, 3), "gbs": round(b / t / 1e9, 1)}
        del bs, g, blk
    tot_t = sum(v["us"] for v in res.values())
    tot_b = sum(l.N * l.K // 32 * 18 + 2 * l.K + 2 * l.N for l in workloads.LLAMA3_8B)
    res["five_shapes"] = {"us": round(tot_t, 2), "gbs": round(tot_b / tot_t / 1e3, 1)}
    out["q4_0_blocks"] = res
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world):
    import w4a16_weight_only_gemm_gb300 as w4
    from w4a16_weight_only_gemm_gb300 import build
    build.build()
    dev = torch.cuda.current_device()
    layers = [make_layer(lin, "llama3_8b_decode", i, keep_rows=PARITY_ROWS if rank == 0 else 0)
              for i, lin in enumerate(workloads.LLAMA3_8B)]
    step_bytes = sum(workloads.algorithmic_bytes(1, lin.N, lin.K) for lin in workloads.LLAMA3_8B)
    stream = torch.cuda.Stream()

    def step():
        for layer in layers:
            gemm_call(layer)

    def steps_fn(n):
        def fn():
            for _ in range(n):
                step()
        return fn
    # STEPS_PER_GRAPH steps per graph replay (a remainder graph makes the
    # count exact): consecutive steps then chain through programmatic
    # dependent launch as eager calls do, not through a graph boundary.
    chunk = min(STEPS_PER_GRAPH, args.steps)
    g = capture(steps_fn(chunk), stream)
    n_full, rem = divmod(args.steps, chunk)
    g_rem = capture(steps_fn(rem), stream) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(-(-max(3, args.warmup) // chunk)):
            g.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(n_full):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    del g, g_rem
    # the same step with one graph replay per step, for reference
    g1 = capture(step, stream)
    t_graph1 = time_graph(g1, stream, 200, 5, world)
    del g1
    secs = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    status = w4.device_status()
    ms_per_step = secs / args.steps * 1e3
    value = step_bytes * world / (secs / args.steps) / 1e9

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,0.02) weights with 0.1% x20 outliers, N(0,1) activations)",
        "config": {"workload": WORKLOAD, "global_batch": 1 * world, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2: 383.7 MB of packed weights per step, no flush",
                   "submission": f"CUDA graphs of {STEPS_PER_GRAPH} steps' w4a16_gemm calls "
                                 "(programmatic dependent launch between consecutive calls, "
                                 "within and across steps)",
                   "ms_per_step_one_graph_per_step": round(t_graph1 * 1e3, 5)},
        "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 1),
        "gpu_launches": args.steps * len(layers),
        "clocks": clk,
        "device_status": status,
    }
    peaks = load_peaks()
    per_rank_gbs = value / world
    result["roofline"] = {
        "bound": "hbm", "achieved": round(per_rank_gbs, 1),
        "peak": peaks.get("hbm_gbs", 6800.0), "unit": "GB/s",
        "frac": round(per_rank_gbs / peaks.get("hbm_gbs", 6800.0), 3),
        "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
        "kernel": "gemv_unit_kernel<1, *> + gemv_kernel<1, 2> (all launches of the step)",
        "bytes_per_launch": step_bytes / len(layers),
        "traffic": recorded_traffic(),
    }
    result["e2e"] = e2e_eager(layers, args, world)
    if rank == 0 and not args.skip_extras:
        result["sections"] = extras(layers)
    if rank == 0:
        result["cpu_baseline"], result["parity"] = cpu_baseline(args.cpu_seconds, layers)
    return result


def e2e_eager(layers, args, world):
    """The same step through the Python API, eager, with host buffers: each
    step copies its five activation vectors from pinned host memory (one
    copy: they sit in one buffer), runs the five GEMVs and reads all five
    outputs back to pinned host memory (one copy)."""
    import w4a16_weight_only_gemm_gb300 as w4
    ks = [l["x"].numel() for l in layers]
    ns = [l["y"].numel() for l in layers]
    x_host = torch.cat([l["x"].reshape(-1).cpu() for l in layers]).pin_memory()
    y_host = torch.empty(sum(ns), dtype=torch.float16).pin_memory()
    x_dev = torch.empty(sum(ks), dtype=torch.float16, device="cuda")
    y_dev = torch.empty(sum(ns), dtype=torch.float16, device="cuda")
    xs = list(torch.split(x_dev, ks))
    ys = list(torch.split(y_dev, ns))
    h2d = x_host.numel() * 2
    d2h = y_host.numel() * 2

    def step():
        x_dev.copy_(x_host, non_blocking=True)
        for l, x, y in zip(layers, xs, ys):
            w4.gemm(x.view(1, -1), l["r"], l["s"], out=y.view(1, -1))
        y_host.copy_(y_dev, non_blocking=True)
    steps = max(10, min(args.steps, 500))
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    barrier(world)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    torch.cuda.synchronize()
    secs = max_over_ranks(start.elapsed_time(end) / 1e3, world) / steps
    step_bytes = sum(workloads.algorithmic_bytes(1, l["lin"].N, l["lin"].K) for l in layers)
    return {"value": round(step_bytes * world / secs / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(secs * 1e3, 4), "steps": steps,
            "how": "eager Python API calls (ctypes -> w4a16_gemm); per step one pinned-host copy of the five "
                   "activation vectors in and one of the five outputs out"}


def extras(layers):
    out = {}
    out["per_shape_m1"] = {lin.name: per_shape_us(lin, "llama3_8b_decode", i)
                           for i, lin in enumerate(workloads.LLAMA3_8B)}
    out["gemv_4096_m1"] = per_shape_us(workloads.SINGLE_GEMV, "gemv_4096", 0)
    out["stack_8b"] = stack_8b()
    sweep = {}
    shapes = [("llama", l) for l in workloads.LLAMA3_8B] + [("qwen", l) for l in workloads.QWEN25_7B]
    for M in workloads.DECODE_SWEEP_M:
        for i, (fam, lin) in enumerate(shapes):
            sweep[f"{fam}_{lin.name}_m{M}"] = per_shape_us(lin, "decode_sweep", i, M=M, reps=10)
    out["decode_sweep"] = sweep
    out["quantizer"] = quantizer_throughput()
    out["prefill_m512"] = prefill()
    out["formats_m1"] = formats_m1()
    out["formats_prefill_m512"] = formats_prefill()
    return out


def prefill():
    """M = 512 prompt pass on the two prefill shapes (tcgen05 path), with a
    cuBLAS fp16 GEMM on pre-dequantised weights of the same shape as the
    practical ceiling (context only)."""
    import w4a16_weight_only_gemm_gb300 as w4
    out = {}
    peaks = load_peaks()
    for i, lin in enumerate(workloads.PREFILL):
        layer = make_layer(lin, "prefill", i, M=workloads.PREFILL_M)
        stream = torch.cuda.Stream()
        g = capture(lambda: gemm_call(layer), stream)
        t = time_graph(g, stream, 20, 3)
        flops = 2.0 * workloads.PREFILL_M * lin.N * lin.K
        wd = torch.randn(lin.N, lin.K, device="cuda", dtype=torch.float16)
        gc = capture(lambda: torch.matmul(layer["x"], wd.t()), stream)
        tc = time_graph(gc, stream, 20, 3)
        tf = flops / t / 1e12
        out[lin.name] = {"us": round(t * 1e6, 2), "tflops": round(tf, 1),
                         "frac_of_measured_bf16_peak": round(tf / peaks.get("bf16_tflops", 1900.0), 3),
                         "cublas_fp16_us": round(tc * 1e6, 2),
                         "cublas_fp16_tflops": round(flops / tc / 1e12, 1)}
        del layer, wd, g, gc
    return out


def formats_prefill():
    """M = 512 prompt pass on the two prefill shapes for format variants of
    w4a16_gemm_ex (tcgen05 path with the variants' dequantisers): group-32
    asymmetric, per-channel symmetric, and group-128 symmetric codes with an
    AWQ activation scale."""
    import w4a16_weight_only_gemm_gb300 as w4
    out = {}
    peaks = load_peaks()
    M = workloads.PREFILL_M
    stream = torch.cuda.Stream()
    for name, group, asym, awq in (("g32_asym", 32, True, False),
                                   ("per_channel_sym", w4.PER_CHANNEL, False, False),
                                   ("g128_sym_awq", 128, False, True)):
        res = {}
        for i, lin in enumerate(workloads.PREFILL):
            sw, sx = synthetic.seeds("prefill", i)
            W = synthetic.master_weight(lin.N, lin.K, sw, device="cuda")
            q, sc, z = w4.quantize_ex(W, group, asymmetric=asym)
            r = w4.repack(q)
            del W, q
            x = synthetic.activations(M, lin.K, sx, device="cuda")
            alpha = (torch.rand(lin.K, device="cuda") * 1.5 + 0.5).half() if awq else None
            y = torch.empty((M, lin.N), dtype=torch.float16, device="cuda")
            g = capture(lambda: w4.gemm_ex(x, r, sc, z, group, out=y, alpha=alpha), stream)
            t = time_graph(g, stream, 20, 3)
            tf = 2.0 * M * lin.N * lin.K / t / 1e12
            plan = w4.gemm_ex_plan(M, lin.N, lin.K, group, asym, awq)
            res[lin.name] = {"us": round(t * 1e6, 2), "tflops": round(tf, 1),
                             "frac_of_measured_bf16_peak": round(tf / peaks.get("bf16_tflops", 1900.0), 3),
                             "cluster": plan["splits"], "ctas": plan["ctas"]}
            del g, r, sc, z, x, y
        out[name] = res
        torch.cuda.empty_cache()
    return out


def stack_8b():
    """Decode tokens of the 8B linear stack: 32 x (QKV, O, gate/up, down)
    + lm_head per token, every matrix distinct (3.87 GB), STEPS_PER_GRAPH
    tokens per CUDA graph replay (consecutive tokens chain through
    programmatic dependent launch, as eager calls do)."""
    lins = workloads.stack_8b()
    layers = [make_layer(lin, "stack_8b", i) for i, lin in enumerate(lins)]
    stream = torch.cuda.Stream()

    def tokens():
        for _ in range(STEPS_PER_GRAPH):
            for l in layers:
                gemm_call(l)
    g = capture(tokens, stream)
    t = time_graph(g, stream, 10, 3) / STEPS_PER_GRAPH
    b = sum(workloads.algorithmic_bytes(1, l.N, l.K) for l in lins)
    del layers, g
    torch.cuda.empty_cache()
    return {"ms_per_token": round(t * 1e3, 4), "tokens_per_s": round(1 / t, 1),
            "gbs": round(b / t / 1e9, 1), "bytes_per_token": b, "gemv_calls": len(lins),
            "tokens_per_graph_replay": STEPS_PER_GRAPH}


def quantizer_throughput():
    import w4a16_weight_only_gemm_gb300 as w4
    N, K = workloads.QUANTIZER_SHAPE
    copies = 4
    Ws = [synthetic.master_weight(N, K, 4000 + i, device="cuda") for i in range(copies)]
    qs = [torch.empty((N, K // 2), dtype=torch.uint8, device="cuda") for _ in range(copies)]
    ss = [torch.empty((N, K // 128), dtype=torch.float16, device="cuda") for _ in range(copies)]
    lib = __import__("w4a16_weight_only_gemm_gb300._native", fromlist=["lib"]).lib()
    stream = torch.cuda.Stream()

    def body():
        sp = torch.cuda.current_stream().cuda_stream
        for W, q, s in zip(Ws, qs, ss):
            rc = lib.w4a16_quantize(W.data_ptr(), N, K, 128, q.data_ptr(), s.data_ptr(), sp)
            assert rc == 0
    g = capture(body, stream)
    t = time_graph(g, stream, 10, 2) / copies
    b = N * K * 2 + N * K // 2 + 2 * N * (K // 128)
    rt = w4.repack(qs[0])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(10):
        w4.repack(qs[0])
    torch.cuda.synchronize()
    trep = (time.perf_counter() - t0) / 10
    del Ws, qs, ss, rt
    return {"us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1), "bytes": b,
            "repack_us_wall": round(trep * 1e6, 1)}


def kernel_sha1() -> str:
    import hashlib
    h = hashlib.sha1()
    for name in ("gemv.cu", "common.cuh"):
        with open(os.path.join(ROOT, "w4a16_weight_only_gemm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram read + write bytes per launch of the GEMV kernel from the committed
    ncu summary, or None if the kernel sources changed since that capture."""
    import re
    path = os.path.join(ROOT, "profiles", "gemv_kernel_llama3_8b_decode_m1.md")
    try:
        text = open(path, encoding="utf-8").read()
    except OSError:
        return None
    sha = re.search(r"kernel_sha1: ([0-9a-f]+)", text)
    tr = re.search(r"traffic_bytes_per_step: (\d+)", text)
    if not sha or not tr or sha.group(1) != kernel_sha1():
        return None
    return int(tr.group(1)) / len(workloads.LLAMA3_8B)


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------
def oracle_inputs(rows_per_shape: int = 64):
    """Sampled rows of each decode shape at M = 1, ready for the oracle:
    (shape, packed rows, scale rows, x).  Packed bytes and scales are random
    (the oracle's cost does not depend on the values)."""
    rng = np.random.default_rng(0)
    prepared = []
    for i, lin in enumerate(workloads.LLAMA3_8B):
        _, sx = synthetic.seeds("llama3_8b_decode", i)
        q = rng.integers(0, 256, size=(rows_per_shape, lin.K // 2), dtype=np.uint8)
        s = rng.uniform(1e-3, 1e-2, size=(rows_per_shape, lin.K // 128)).astype(np.float16)
        x = synthetic.activations(1, lin.K, sx).view(torch.int16).numpy().view(np.uint16)
        prepared.append((lin, q, s.view(np.uint16), x))
    return prepared


def oracle_pass(prepared, keep: bool = False):
    """One pass of the oracle over the sampled rows; returns algorithmic bytes
    of the work done (packed rows + their scales + x + the outputs), or with
    keep=True the outputs themselves."""
    import oracle
    done, ys = 0, []
    for lin, q, s, x in prepared:
        rows = np.arange(q.shape[0])
        y = oracle.gemm_rows(x, q, s, rows)
        if keep:
            ys.append(y)
        done += q.shape[0] * (lin.K // 2 + 2 * (lin.K // 128) + 2) + 2 * lin.K
    return ys if keep else done


ORACLE_SAMPLE = ("{rows} sampled rows of each of the 5 decode shapes (M=1) per pass; "
                 "binary64 oracle, OpenMP over rows")


def cpu_baseline(seconds: float, layers):
    """The oracle timed on the host cores over the timed layers' sampled rows
    (their master-weight rows quantized by the oracle itself, the layers' own
    activations), and -- as a by-product, outside any timed region -- the
    parity of the GPU outputs of the last timed step at those rows."""
    import oracle
    prepared = []
    for l in layers:
        w16 = l["W_rows"].contiguous().view(torch.int16).numpy().view(np.uint16)
        q, s = oracle.quantize(w16)
        x = l["x"].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
        prepared.append((l["lin"], q, s, x))
    ys = oracle_pass(prepared, keep=True)
    worst_max, worst_l2 = 0.0, 0.0
    for l, y_ref in zip(layers, ys):
        y = l["y"][:, torch.from_numpy(l["rows"]).cuda()].float().cpu().numpy().astype(np.float64)
        err = np.abs(y - y_ref)
        worst_max = max(worst_max, float(err.max() / np.abs(y_ref).max()))
        worst_l2 = max(worst_l2, float(np.linalg.norm(err) / np.linalg.norm(y_ref)))
    parity = {"rows_per_layer": len(layers[0]["rows"]), "layers": len(layers),
              "max_rel": round(worst_max, 6), "l2": round(worst_l2, 6),
              "bar": {"max_rel": 2e-3, "l2": 1e-3},
              "pass": bool(worst_max <= 2e-3 and worst_l2 <= 1e-3),
              "how": "GPU y of the last timed step at sampled rows vs the binary64 oracle on the "
                     "oracle's own quantization of the same master-weight rows (worst layer)"}
    done, passes = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        done += oracle_pass(prepared)
        passes += 1
    secs = time.perf_counter() - t0
    rows = len(layers[0]["rows"])
    base = {"value": round(done / secs / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"{passes} passes: " + ORACLE_SAMPLE.format(rows=rows),
            "seconds": round(secs, 2)}
    return base, parity


def run_reference(args, rank, world):
    """The CPU oracle on the headline workload: each step is one pass over a
    bounded sample (64 rows of each decode shape), timed on the host cores."""
    import oracle
    if rank != 0:
        return None
    prepared = oracle_inputs(64)
    for _ in range(args.warmup):
        oracle_pass(prepared)
    done = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        done += oracle_pass(prepared)
    secs = time.perf_counter() - t0
    value = done / secs / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle.num_threads(),
                         "sample": "per step: " + ORACLE_SAMPLE.format(rows=64)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.section is not None:
        from w4a16_weight_only_gemm_gb300 import build
        build.build()
        run = {"prefill": prefill, "quantizer": quantizer_throughput, "stack": stack_8b,
               "formats": formats_m1, "formats_prefill": formats_prefill,
               "per_shape": lambda: {lin.name: per_shape_us(lin, "llama3_8b_decode", i)
                                     for i, lin in enumerate(workloads.LLAMA3_8B)}}
        print(json.dumps({"section": args.section, "result": run[args.section]()}), flush=True)
        return
    if args.impl == "reference":
        # Only rank 0 times the CPU oracle; other ranks exit without work.
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        res = run_reference(args, rank, world)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world = dist_init(args.gpus)
    res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
