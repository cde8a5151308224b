#!/usr/bin/env python3
"""Benchmark of the W4A16 group-quantized linear layer on one GB300.

Metric: achieved HBM GB/s (algorithmic bytes / time) of the W4A16-g128 GEMM,
with TFLOP/s and the fraction of the roofline beside it. A step is one pass
over every linear layer of the workload at every batch size M of it (the
Llama-2-7B decode workload by default: qkv, o_proj, gate_up, down at
M = 1, 4, 8, 16), with the packed weights resident in HBM and rotated over
enough copies that the working set exceeds L2 between repeats.

Algorithmic bytes of one GEMM = K*N/2 (int4 codes) + 2*G*N (fp16 scales)
+ G*N/2 (int4 zero points) + 2*M*K (A) + 2*M*N (Y), G = K/group.
Roofline time = max(bytes / HBM peak, 2*M*N*K / fp16 tensor peak).

  python bench.py [--steps K] [--warmup W] [--workload 1] [--sweep out.jsonl]
  python bench.py --act bf16|a8 ...      # bf16 activations, or W4A8
  python bench.py --impl reference ...   # the CPU oracle on the same metric

The end-to-end figure (`e2e`) runs the same step through the public API with
every step's input copied in from pinned host memory and its result copied
back, double-buffered on a second stream as a serving loop would (step i
overlaps step i+1's input copy and step i-1's result copy).

Under torchrun (WORLD_SIZE > 1) every rank runs its own replica of the
workload on its own GPU (independent problems, no collective on the data
path); the step time is the maximum over ranks and the value is the total
over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- accounting

def alg_bytes(M, K, N, group):
    G = K // group
    return K * N // 2 + 2 * G * N + G * N // 2 + 2 * M * K + 2 * M * N


def flops(M, K, N):
    return 2 * M * N * K


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "tflops": float(p["bf16_tflops"]),
                "tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_PEAKS["hbm_gbs"], "tflops": FALLBACK_PEAKS["bf16_tflops"],
            "tflops_sustained": FALLBACK_PEAKS["bf16_tflops_sustained"], "source": "fallback"}


# ncu summaries under profiles/: the dominant kernel of a workload, the sources
# that build it, and the summary holding its DRAM bytes per launch
PROFILED = {
    1: ("decode_resident_kernel", ["decode_impl.cuh", "decode.cu", "common.cuh"],
        "decode_resident_kernel_llama2-7b-decode.md"),
    3: ("tc_gemm_kernel", ["tc_gemm.cu", "common.cuh"], "tc_gemm_kernel_llama2-7b-prefill.md"),
}


def profiled_traffic(workload):
    """DRAM bytes per launch (read + write) of the workload's dominant kernel
    from its committed ncu summary, or None if there is none or the kernel's
    sources have changed since the counters were taken."""
    import hashlib
    if workload not in PROFILED:
        return None
    _, srcs, summary = PROFILED[workload]
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in srcs:
        with open(os.path.join(ROOT, "bit_weight_only_g128_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    fields = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith(("#", " ", "|")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    sha = next((v for k, v in fields.items() if k.startswith("kernel source sha256")), None)
    if sha != h.hexdigest()[:16]:
        return None
    try:
        return float(fields["traffic per launch (bytes)"])
    except (KeyError, ValueError):
        return None


def roofline_us(M, K, N, group, pk):
    t_mem = alg_bytes(M, K, N, group) / (pk["hbm_gbs"] * 1e9)
    t_tc = flops(M, K, N) / (pk["tflops"] * 1e12)
    return 1e6 * max(t_mem, t_tc), ("hbm" if t_mem >= t_tc else "tensor")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if "Active" in v
                          and "Not" not in v})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------- distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return None, 0, 1, 0
    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return dist, dist.get_rank(), world, local


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle

def oracle_sample_pass(wl, ncols, group_cache):
    """One pass of the oracle over every case of the workload, restricted to
    the first `ncols` output columns of each layer. Returns (seconds, bytes, flops)."""
    import oracle
    secs, nbytes, nflops = 0.0, 0, 0
    for (layer, M, K, N, g) in wl.cases():
        n = min(ncols, N)
        key = (layer, K, N, g, n)
        if key not in group_cache:
            W = synthetic.weights(wl.cfg, K, N)[:, :n]
            group_cache[key] = oracle.quantize(np.ascontiguousarray(W), g)
        q, s, z = group_cache[key]
        A = synthetic.activations(wl.cfg, M, K, N, outliers=wl.outliers)
        t0 = time.perf_counter()
        deq = oracle.dequantize(q, s, z, g)
        oracle.matmul(A, deq)
        secs += time.perf_counter() - t0
        G = K // g
        nbytes += K * n // 2 + 2 * G * n + G * n // 2 + 2 * M * K + 2 * M * n
        nflops += 2 * M * n * K
    return secs, nbytes, nflops


def cpu_baseline(wl, target_s=15.0):
    import oracle
    cache = {}
    probe_cols = 64
    t, _, _ = oracle_sample_pass(wl, probe_cols, cache)
    ncols = max(16, int(probe_cols * target_s / max(t, 1e-3)) // 16 * 16)
    ncols = min(ncols, max(N for (_, _, _, N, _) in wl.cases()))
    t, b, f = oracle_sample_pass(wl, ncols, cache)
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
            "tflops": f / t / 1e12, "seconds": t,
            "sample": (f"every GEMM of one step ({len(wl.cases())} cases) restricted to the "
                       f"first {ncols} output columns of each layer; dequantize + fp64 matmul")}


def workload_config(wl):
    """The `config` object of the JSON line (both arms)."""
    return {"workload": wl.name,
            "layers": [f"{n} K={k} N={nn}" for (n, k, nn) in wl.layers],
            "M": list(wl.ms), "group": list(wl.groups),
            "gemms_per_step": len(wl.cases())}


def run_reference(args, wl, dist, rank, world):
    """The CPU oracle as the reference arm, on the same metric and workload."""
    if rank != 0:
        return
    import oracle
    budget = 150.0 / max(1, args.steps + args.warmup)
    cache = {}
    t, _, _ = oracle_sample_pass(wl, 32, cache)
    ncols = max(16, int(32 * budget / max(t, 1e-3)) // 16 * 16)
    for _ in range(args.warmup):
        oracle_sample_pass(wl, ncols, cache)
    tot_s, tot_b = 0.0, 0
    for _ in range(args.steps):
        s, b, _ = oracle_sample_pass(wl, ncols, cache)
        tot_s += s
        tot_b += b
    value = tot_b / tot_s / 1e9
    sample = (f"each step: every GEMM of the workload restricted to the first {ncols} output "
              f"columns of each layer (dequantize + fp64 matmul)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm

METRIC = "W4A16-g128 GEMM HBM GB/s (algorithmic bytes / time), % of roofline, 1 GB300"


# extra keyword arguments of every timed gemm call (W4A8: {"a8": True})
GEMM_KW = {}


class Case:
    def __init__(self, layer, M, K, N, group):
        self.layer, self.M, self.K, self.N, self.group = layer, M, K, N, group

    @property
    def key(self):
        return (self.layer, self.K, self.N, self.group)


def _aligned_views(torch, shapes, dtype, device):
    """One flat buffer holding several tensors, each 256-byte aligned."""
    esize = torch.tensor([], dtype=dtype).element_size()
    align = 256 // esize
    offs, total = [], 0
    for shp in shapes:
        offs.append(total)
        total += (math.prod(shp) + align - 1) // align * align
    flat = torch.zeros(max(total, 1), dtype=dtype, device=device)
    return flat, [flat[o:o + math.prod(s)].view(*s) for o, s in zip(offs, shapes)]


def build_gpu_workload(wl, torch, w4, device, copies=None, act="f16"):
    cases = [Case(*c) for c in wl.cases()]
    layers = {}
    for c in cases:
        if c.key not in layers:
            W = torch.from_numpy(synthetic.weights(wl.cfg, c.K, c.N)).to(device)
            layers[c.key] = w4.quantize_pack(W, c.group)
            del W
    packed_bytes = sum(pw.nbytes for pw in layers.values())
    if copies is None:
        copies = max(2, math.ceil(3 * L2_BYTES / packed_bytes))
    rot = [layers]
    for _ in range(copies - 1):
        rot.append({k: w4.PackedWeight(pw.Wq.clone(), pw.Sp.clone(), pw.Zp.clone(), pw.K, pw.N,
                                       pw.group) for k, pw in layers.items()})
    # activations and results: fp16, or bf16 (the fp16 inputs rounded to bf16)
    adt = torch.bfloat16 if act == "bf16" else torch.float16
    a_flat, a_views = _aligned_views(torch, [(c.M, c.K) for c in cases], adt, device)
    y_flat, y_views = _aligned_views(torch, [(c.M, c.N) for c in cases], adt, device)
    # one workspace serves every call: they run one after another on one stream
    ws = w4.new_workspace(max(w4.workspace_size(c.M, c.N, c.K, c.group, **GEMM_KW) for c in cases),
                          device)
    for r in rot:
        r["workspace"] = ws
    for c, av in zip(cases, a_views):
        av.copy_(torch.from_numpy(synthetic.activations(wl.cfg, c.M, c.K, c.N,
                                                        outliers=wl.outliers)))
    return cases, rot, (a_flat, a_views), (y_flat, y_views), packed_bytes


def sanity_check(wl, cases, rot, a_views, y_views, torch, w4):
    """Sampled columns of every distinct layer against the oracle (not timed)."""
    import oracle
    seen = set()
    for c, A, Y in zip(cases, a_views, y_views):
        if c.key in seen:
            continue
        seen.add(c.key)
        w4.gemm(A, rot[0][c.key], out=Y, workspace=rot[0]["workspace"], **GEMM_KW)
        torch.cuda.synchronize()
        cols = synthetic.sample_indices(c.N, 32, seed=0, salt=c.N)
        W = synthetic.weights(wl.cfg, c.K, c.N)[:, cols]
        q, s, z = oracle.quantize(np.ascontiguousarray(W), c.group)
        got = np.ascontiguousarray(Y.cpu().view(torch.int16).numpy().view(np.uint16)[:, cols])
        a_bits = A.cpu().view(torch.int16).numpy().view(np.uint16)
        if GEMM_KW.get("a8"):
            vals = (oracle.from_bf16 if A.dtype == torch.bfloat16 else oracle.from_half)(a_bits)
            aq, sa = oracle.quantize_act(vals)
            y, mag = oracle.reference_a8(aq, sa, q, s, z, c.group)
            ratio, _ = (oracle.check_bf16 if A.dtype == torch.bfloat16 else oracle.check)(got, y, mag)
        elif A.dtype == torch.bfloat16:
            y, mag = oracle.reference_bf16(a_bits, q, s, z, c.group)
            ratio, _ = oracle.check_bf16(got, y, mag)
        else:
            y, mag = oracle.reference(a_bits, q, s, z, c.group)
            ratio, _ = oracle.check(got, y, mag)
        if not ratio <= 1.0:
            raise SystemExit(f"parity check failed for {c.layer} M={c.M}: err/bound {ratio}")


def capture_step(torch, w4, cases, weights, a_views, y_views, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c, A, Y in zip(cases, a_views, y_views):
            w4.gemm(A, weights[c.key], out=Y, workspace=weights["workspace"], static_weights=True,
                    **GEMM_KW)
    return g


def time_graphs(torch, graphs, steps, stream):
    """Seconds for `steps` graph replays, timed with events on the stream the
    graphs are replayed on (CUDAGraph.replay launches on the current stream)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


def per_case_times(torch, w4, cases, rot, a_views, y_views, stream, reps=20):
    """Average duration of one launch of each case (graph of `reps` launches
    rotating over the weight copies, timed with events)."""
    out = []
    for c, A, Y in zip(cases, a_views, y_views):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                w4.gemm(A, rot[r % len(rot)][c.key], out=Y, workspace=rot[0]["workspace"],
                        static_weights=True, **GEMM_KW)
        time_graphs(torch, [g], 3, stream)
        secs = time_graphs(torch, [g], 5, stream) / (5 * reps)
        out.append(secs)
        del g
    return out


def silu_mul_times(torch, w4, cases, rot, a_views, stream, reps=20):
    """Average launch time of each gate_up case with the fused gate/up
    epilogue (output [M, N/2] = silu(gate) * up), timed like per_case_times."""
    out = []
    for c, A in zip(cases, a_views):
        if c.layer != "gate_up":
            continue
        Y = torch.empty((c.M, c.N // 2), dtype=A.dtype, device=A.device)
        ws = w4.new_workspace(w4.workspace_size(c.M, c.N, c.K, c.group, silu_mul=True, **GEMM_KW),
                              A.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                w4.gemm(A, rot[r % len(rot)][c.key], out=Y, workspace=ws, static_weights=True,
                        silu_mul=True, **GEMM_KW)
        time_graphs(torch, [g], 3, stream)
        out.append((c, time_graphs(torch, [g], 5, stream) / (5 * reps)))
        del g, ws
    return out


def roofline_entry(args, pk, cases, step_bytes, step_flops, secs):
    """Roofline of the step's kernel launches: bound by HBM if the step's
    algorithmic bytes take longer at the measured copy bandwidth than its
    flops at the measured dense tensor rate (fp16 runs at the bf16 rate),
    else by the tensor cores. achieved = algorithmic bytes (or flops) per
    launch / mean launch time; traffic = ncu DRAM bytes per launch."""
    t_mem = step_bytes / (pk["hbm_gbs"] * 1e9)
    t_tc = step_flops / (pk["tflops"] * 1e12)
    per_launch_s = secs / args.steps / len(cases)
    kernel = PROFILED.get(args.workload, ("decode_kernel" if t_mem >= t_tc else "tc_gemm_kernel",))[0]
    entry = {"traffic": profiled_traffic(args.workload),
             "traffic_unit": "DRAM bytes per launch (ncu summary in profiles/)",
             "algorithmic_bytes_per_launch": step_bytes / len(cases),
             "peak_source": pk["source"], "kernel": kernel}
    if t_mem >= t_tc:
        achieved = step_bytes / len(cases) / per_launch_s / 1e9
        entry.update({"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                      "frac": achieved / pk["hbm_gbs"]})
    else:
        achieved = step_flops / len(cases) / per_launch_s / 1e12
        entry.update({"bound": "tensor", "achieved": achieved, "peak": pk["tflops"],
                      "unit": "TFLOP/s", "frac": achieved / pk["tflops"]})
    return entry


def run_ours(args, wl, dist, rank, world, local):
    import torch
    import bit_weight_only_g128_gb300 as w4

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.act == "a8":
        GEMM_KW["a8"] = True
    pk = peaks()
    cases, rot, (a_flat, a_views), (y_flat, y_views), packed_bytes = build_gpu_workload(
        wl, torch, w4, device, args.copies, "bf16" if args.act == "bf16" else "f16")
    sanity_check(wl, cases, rot, a_views, y_views, torch, w4)

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    graphs = [capture_step(torch, w4, cases, r, a_views, y_views, stream) for r in rot]
    step_bytes = sum(alg_bytes(c.M, c.K, c.N, c.group) for c in cases)
    step_flops = sum(flops(c.M, c.K, c.N) for c in cases)
    step_roof_us = sum(roofline_us(c.M, c.K, c.N, c.group, pk)[0] for c in cases)

    time_graphs(torch, graphs, args.warmup, stream)
    barrier(dist)
    with ClockSampler(local) as clk:
        secs = time_graphs(torch, graphs, args.steps, stream)
    barrier(dist)
    secs = max_over_ranks(dist, secs)
    clocks = clk.summary()

    # end to end through the public API: every step's activations copied in
    # from pinned host memory and every step's results read back (weights are
    # resident model state). The copies are double-buffered on a second
    # stream, as a serving loop would run them: during step i the next step's
    # input goes in and the previous step's result comes out, and the timed
    # region also holds the first step's input copy and the last step's
    # result copy.
    a_host = torch.empty_like(a_flat, device="cpu").pin_memory()
    a_host.copy_(a_flat)
    y_host = torch.empty_like(y_flat, device="cpu").pin_memory()
    a_flat2, a_views2 = _aligned_views(torch, [(c.M, c.K) for c in cases], a_flat.dtype, device)
    y_flat2, y_views2 = _aligned_views(torch, [(c.M, c.N) for c in cases], y_flat.dtype, device)
    a_bufs, y_bufs = (a_flat, a_flat2), (y_flat, y_flat2)
    a_sets, y_sets = (a_views, a_views2), (y_views, y_views2)
    io = torch.cuda.Stream(device)
    e2e_graphs = {}
    for b in (0, 1):
        for ri, r in enumerate(rot):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fork = torch.cuda.Event()
                fork.record(stream)
                io.wait_event(fork)
                with torch.cuda.stream(io):
                    a_bufs[1 - b].copy_(a_host, non_blocking=True)   # the next step's input
                    y_host.copy_(y_bufs[1 - b], non_blocking=True)   # the previous step's result
                join = torch.cuda.Event()
                join.record(io)
                for c, A, Y in zip(cases, a_sets[b], y_sets[b]):
                    w4.gemm(A, r[c.key], out=Y, workspace=r["workspace"], static_weights=True,
                            **GEMM_KW)
                stream.wait_event(join)
            e2e_graphs[(b, ri)] = g

    def time_e2e(steps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            a_bufs[0].copy_(a_host, non_blocking=True)       # the first step's input
            for i in range(steps):
                e2e_graphs[(i % 2, i % len(rot))].replay()
            y_host.copy_(y_bufs[(steps - 1) % 2], non_blocking=True)  # the last step's result
            end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / 1e3

    time_e2e(args.warmup)
    barrier(dist)
    e2e_secs = max_over_ranks(dist, time_e2e(args.steps))

    value = world * step_bytes * args.steps / secs / 1e9
    e2e_value = world * step_bytes * args.steps / e2e_secs / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.act,
        "data": "synthetic",
        "config": {**workload_config(wl),
                   "activations": args.act,
                   "static_weights": True,
                   "l2": (f"inputs larger than L2: {len(rot)} rotating copies of the packed "
                          f"weights, {len(rot) * packed_bytes / 2**20:.0f} MiB")},
        "tflops": world * step_flops * args.steps / secs / 1e12,
        "roofline_frac_step": step_roof_us * 1e-6 * args.steps / secs,
        "roofline": roofline_entry(args, pk, cases, step_bytes, step_flops, secs),
        "e2e": {"value": e2e_value, "unit": "GB/s",
                "copies": "double-buffered on a second stream: step i overlaps the input copy "
                          "of step i+1 and the result copy of step i-1",
                "h2d_bytes_per_step": sum(2 * c.M * c.K for c in cases),
                "d2h_bytes_per_step": sum(2 * c.M * c.N for c in cases)},
        # one kernel per GEMM (W4A8: the activation quantization too)
        "gpu_launches": len(cases) * args.steps * (2 if GEMM_KW.get("a8") else 1),
        "clocks": clocks,
    }
    if args.sweep:
        times = per_case_times(torch, w4, cases, rot, a_views, y_views, stream)
        with open(args.sweep, "a") as f:
            for c, t in zip(cases, times):
                roof, bound = roofline_us(c.M, c.K, c.N, c.group, pk)
                path, parts = w4.plan(c.M, c.N, c.K, c.group)
                f.write(json.dumps({
                    "workload": wl.name, "act": args.act, "layer": c.layer, "M": c.M, "K": c.K,
                    "N": c.N, "group": c.group, "path": path, "parts": parts, "us": 1e6 * t,
                    "GBps": alg_bytes(c.M, c.K, c.N, c.group) / t / 1e9,
                    "TFLOPs": flops(c.M, c.K, c.N) / t / 1e12, "roofline_us": roof,
                    "bound": bound, "frac": roof / (1e6 * t)}) + "\n")
            for c, t in silu_mul_times(torch, w4, cases, rot, a_views, stream):
                # the fused layer writes half the columns
                nbytes = alg_bytes(c.M, c.K, c.N, c.group) - c.M * c.N
                f.write(json.dumps({
                    "workload": wl.name, "act": args.act, "layer": "gate_up+silu_mul", "M": c.M, "K": c.K,
                    "N": c.N, "group": c.group, "us": 1e6 * t, "GBps": nbytes / t / 1e9,
                    "TFLOPs": flops(c.M, c.K, c.N) / t / 1e12}) + "\n")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=1, help="workload index (0..4)")
    ap.add_argument("--copies", type=int, default=None, help="weight copies for L2 rotation")
    ap.add_argument("--sweep", default=None, help="append per-case timings (JSONL) here")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--act", choices=("f16", "bf16", "a8"), default="f16",
                    help="activations: fp16, bf16 (W4A16_BF16) or fp16 quantized to int8 per "
                         "row inside each call (W4A8, W4A16_ACT_A8); the same weights")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    wl = synthetic.workload(args.workload)
    dist, rank, world, local = dist_init()
    try:
        if args.impl == "reference":
            run_reference(args, wl, dist, rank, world)
        else:
            run_ours(args, wl, dist, rank, world, local)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
