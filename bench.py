#!/usr/bin/env python3
"""Benchmark of the W4A16 group-quantized linear layer on one GB300.

Metric: W4A16 GEMM TFLOP/s and HBM GB/s against M, and the fraction of the
roofline. A step is one pass over every linear layer of the workload at every
batch size M of it, with the packed weights resident in HBM and rotated over
enough copies that the working set exceeds L2 between repeats. The default
workload is the Llama-2-70B sweep: qkv, o_proj, gate_up, down at
M = 1, 8, 64, 512, 4096, with groups of 128 and per-channel groups (group = K),
40 GEMMs per step.

Algorithmic bytes of one GEMM = K*N/2 (int4 codes) + 2*G*N (fp16 scales)
+ G*N/2 (int4 zero points) + 2*M*K (A) + 2*M*N (Y), G = K/group; FLOPs =
2*M*N*K. Roofline time = max(bytes / HBM peak, FLOPs / 16-bit tensor peak).

The step runs as two CUDA graphs, timed separately with events on the stream
they replay on: the GEMMs whose roofline is HBM-bound, then those that are
tensor-bound. `value` is the step's TFLOP/s (GB/s when the step's roofline
time is mostly HBM-bound); `roofline` describes the dominant group's kernel,
and `roofline_by_bound` both groups.

  python bench.py [--steps K] [--warmup W] [--workload 4] [--sweep out.jsonl]
  python bench.py --act bf16|a8 ...      # bf16 activations, or W4A8
  python bench.py --impl reference ...   # the CPU oracle on the same metric

The end-to-end figure (`e2e`) runs the same step through the public API with
every step's input copied in from pinned host memory and its result copied
back, double-buffered on two more streams (one per copy direction) as a
serving loop would (step i overlaps step i+1's input copy and step i-1's
result copy).

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
    2: ("tc_gemm_kernel", ["tc_gemm.cu", "tc_ptx.cuh", "common.cuh"], "tc_gemm_kernel_llama2-13b-mid.md"),
    3: ("tc_pair_kernel", ["tc_pair.cu", "tc_gemm.cu", "tc_ptx.cuh", "common.cuh"],
        "tc_pair_kernel_llama2-7b-prefill.md"),
    4: ("tc_pair_kernel", ["tc_pair.cu", "tc_gemm.cu", "tc_ptx.cuh", "common.cuh"],
        "tc_pair_kernel_llama2-70b-sweep.md"),
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


def headline_unit(wl, pk):
    """TFLOP/s when the step's roofline time is mostly tensor-bound, else GB/s."""
    t_mem = t_tc = 0.0
    for (_, M, K, N, g) in wl.cases():
        t, bound = roofline_us(M, K, N, g, pk)
        if bound == "hbm":
            t_mem += t
        else:
            t_tc += t
    return "TFLOP/s" if t_tc > t_mem else "GB/s"


def rate(unit, nbytes, nflops, secs):
    return nflops / secs / 1e12 if unit == "TFLOP/s" else nbytes / secs / 1e9


def cpu_baseline(wl, unit, target_s=15.0):
    import oracle
    cache = {}
    probe_cols = 16
    t, _, _ = oracle_sample_pass(wl, probe_cols, cache)
    ncols = max(16, int(probe_cols * target_s / max(t, 1e-3)) // 16 * 16)
    ncols = min(ncols, max(N for (_, _, _, N, _) in wl.cases()))
    t, b, f = oracle_sample_pass(wl, ncols, cache)
    return {"value": rate(unit, b, f, t), "unit": unit, "cores": oracle.threads(), "kind": "oracle",
            "gbs": b / t / 1e9, "tflops": f / t / 1e12, "seconds": t,
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
    unit = headline_unit(wl, peaks())
    budget = 150.0 / max(1, args.steps + args.warmup)
    cache = {}
    t, _, _ = oracle_sample_pass(wl, 16, cache)
    ncols = max(16, int(16 * budget / max(t, 1e-3)) // 16 * 16)
    for _ in range(args.warmup):
        oracle_sample_pass(wl, ncols, cache)
    tot_s, tot_b, tot_f = 0.0, 0, 0
    for _ in range(args.steps):
        s, b, f = oracle_sample_pass(wl, ncols, cache)
        tot_s += s
        tot_b += b
        tot_f += f
    value = rate(unit, tot_b, tot_f, tot_s)
    sample = (f"each step: every GEMM of the workload restricted to the first {ncols} output "
              f"columns of each layer (dequantize + fp64 matmul)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm

METRIC = "W4A16-g128 GEMM TFLOP/s and HBM GB/s vs M (1-4096), % of roofline, 1 GB300"

# kernel of each path that w4a16_plan reports
KERNEL_OF_PATH = {"decode-resident": "decode_resident_kernel", "decode-streamk": "decode_kernel",
                  "tensor": "tc_gemm_kernel", "tensor-pair": "tc_pair_kernel"}

# extra keyword arguments of every timed gemm call (W4A8: {"a8": True})
GEMM_KW = {}


class Case:
    def __init__(self, layer, M, K, N, group):
        self.layer, self.M, self.K, self.N, self.group = layer, M, K, N, group

    @property
    def key(self):
        return (self.layer, self.K, self.N, self.group)


def split_by_bound(cases, pk):
    """Indices of the cases whose roofline is HBM-bound, then tensor-bound."""
    hbm, tc = [], []
    for i, c in enumerate(cases):
        (hbm if roofline_us(c.M, c.K, c.N, c.group, pk)[1] == "hbm" else tc).append(i)
    return hbm, tc


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


def capture(torch, w4, cases, idx, weights, a_views, y_views, stream):
    """A CUDA graph of the GEMMs `idx` of one step (None if there are none)."""
    if not idx:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in idx:
            c = cases[i]
            w4.gemm(a_views[i], weights[c.key], out=y_views[i], workspace=weights["workspace"],
                    static_weights=True, **GEMM_KW)
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


def time_split_steps(torch, parts, steps, stream):
    """Run `steps` steps, each the replay of its part graphs in order (parts[r]
    is a list of graphs for rotation copy r, None for an empty part). Events
    on the replay stream bracket every part of every step; returns per-step
    lists of part durations in seconds."""
    nparts = len(parts[0])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nparts + 1)] for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            gs = parts[i % len(parts)]
            ev[i][0].record(stream)
            for j, g in enumerate(gs):
                if g is not None:
                    g.replay()
                ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    return [[ev[i][j].elapsed_time(ev[i][j + 1]) / 1e3 for j in range(nparts)] for i in range(steps)]


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


def group_roofline(pk, cases, idx, secs, steps, bound, kernels):
    """Roofline entry of the launches `idx` of a step that took `secs` in
    total over `steps` steps: achieved = algorithmic bytes (or flops) per
    launch / mean launch time of the group. Tensor-bound launches run back to
    back for the whole timed region, so their peak is the sustained dense
    rate (the burst fraction is given beside it)."""
    n = len(idx) * steps
    per_launch_s = secs / n
    nbytes = sum(alg_bytes(cases[i].M, cases[i].K, cases[i].N, cases[i].group) for i in idx)
    nflops = sum(flops(cases[i].M, cases[i].K, cases[i].N) for i in idx)
    roof_s = sum(roofline_us(cases[i].M, cases[i].K, cases[i].N, cases[i].group, pk)[0]
                 for i in idx) * 1e-6
    entry = {"launches_per_step": len(idx), "kernels": kernels,
             "ms_per_step": 1e3 * secs / steps,
             "algorithmic_bytes_per_launch": nbytes / len(idx),
             "flops_per_launch": nflops / len(idx),
             "roofline_frac": roof_s * steps / secs}
    if bound == "hbm":
        achieved = nbytes / len(idx) / per_launch_s / 1e9
        entry.update({"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                      "frac": achieved / pk["hbm_gbs"], "peak_kind": "copy bandwidth"})
    else:
        achieved = nflops / len(idx) / per_launch_s / 1e12
        entry.update({"bound": "tensor", "achieved": achieved, "peak": pk["tflops_sustained"],
                      "unit": "TFLOP/s", "frac": achieved / pk["tflops_sustained"],
                      "peak_kind": "sustained dense bf16 (16-bit) rate",
                      "frac_of_burst": achieved / pk["tflops"]})
    return entry


def kernels_of(w4, cases, idx):
    """Kernel names (with launch counts) that the automatic plan uses for the
    cases `idx`."""
    out = {}
    for i in idx:
        c = cases[i]
        path, _ = w4.plan(c.M, c.N, c.K, c.group)
        name = KERNEL_OF_PATH.get(path, path)
        out[name] = out.get(name, 0) + 1
    return out


def host_call_us(torch, w4, case, weights, A, Y, stream, calls=200):
    """Host time per eager call (enqueue only: no synchronization inside the
    loop) through the Python API and through the C ABI directly."""
    import ctypes
    lib = w4.lib()
    pw = weights[case.key]
    ws = weights["workspace"]
    flags = w4.STATIC_WEIGHTS | (w4.ACT_A8 if GEMM_KW.get("a8") else 0) | \
        (w4.BF16 if A.dtype == torch.bfloat16 else 0)
    s = ctypes.c_void_p(stream.cuda_stream)
    out = {}
    with torch.cuda.stream(stream):
        for name in ("python", "c_abi"):
            for rep in range(2):          # the first pass warms caches
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                if name == "python":
                    for _ in range(calls):
                        w4.gemm(A, pw, out=Y, workspace=ws, static_weights=True, **GEMM_KW)
                else:
                    args = (A.data_ptr(), pw.Wq.data_ptr(), pw.Sp.data_ptr(), pw.Zp.data_ptr(),
                            case.M, case.N, case.K, case.group, Y.data_ptr(), ws.data_ptr(),
                            ws.numel(), flags, 0, s)
                    for _ in range(calls):
                        rc = lib.w4a16_gemm_ex(*args)
                        if rc != 0:
                            raise RuntimeError(lib.w4a16_last_error().decode())
                t1 = time.perf_counter()
                torch.cuda.synchronize()
            out[name] = 1e6 * (t1 - t0) / calls
    return out


def run_ours(args, wl, dist, rank, world, local):
    import torch
    import bit_weight_only_g128_gb300 as w4

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.act == "a8":
        GEMM_KW["a8"] = True
    pk = peaks()
    unit = headline_unit(wl, pk)
    cases, rot, (a_flat, a_views), (y_flat, y_views), packed_bytes = build_gpu_workload(
        wl, torch, w4, device, args.copies, "bf16" if args.act == "bf16" else "f16")
    sanity_check(wl, cases, rot, a_views, y_views, torch, w4)

    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    hbm_idx, tc_idx = split_by_bound(cases, pk)
    parts = [[capture(torch, w4, cases, hbm_idx, r, a_views, y_views, stream),
              capture(torch, w4, cases, tc_idx, r, a_views, y_views, stream)] for r in rot]
    step_bytes = sum(alg_bytes(c.M, c.K, c.N, c.group) for c in cases)
    step_flops = sum(flops(c.M, c.K, c.N) for c in cases)
    step_roof_us = sum(roofline_us(c.M, c.K, c.N, c.group, pk)[0] for c in cases)

    time_split_steps(torch, parts, args.warmup, stream)
    barrier(dist)
    with ClockSampler(local) as clk:
        per_step = time_split_steps(torch, parts, args.steps, stream)
    barrier(dist)
    secs_parts = [sum(s[j] for s in per_step) for j in range(2)]
    secs = max_over_ranks(dist, sum(secs_parts))
    clocks = clk.summary()
    step_ms = sorted(1e3 * sum(s) for s in per_step)

    groups = {}
    for name, idx, j in (("hbm", hbm_idx, 0), ("tensor", tc_idx, 1)):
        if idx:
            groups[name] = group_roofline(pk, cases, idx, secs_parts[j], args.steps, name,
                                          kernels_of(w4, cases, idx))
    dominant = max(groups, key=lambda k: groups[k]["ms_per_step"])
    roofline = dict(groups[dominant])
    roofline["kernel"] = max(roofline["kernels"], key=roofline["kernels"].get)
    roofline.update({"traffic": profiled_traffic(args.workload),
                     "traffic_unit": "DRAM bytes per launch (ncu summary in profiles/)",
                     "peak_source": pk["source"]})

    # end to end through the public API: every step's activations copied in
    # from pinned host memory and every step's results read back (weights are
    # resident model state). The copies are double-buffered on two more
    # streams, one per direction (host-to-device and device-to-host copies then
    # run at once: 9.0 against 13.0 ms for 1 GB in and 1.6 GB out on GB300), as
    # a serving loop would run them: during step i the next step's input goes
    # in and the previous step's result comes out, and the timed region also
    # holds the first step's input copy and the last step's result copy.
    a_host = torch.empty_like(a_flat, device="cpu").pin_memory()
    a_host.copy_(a_flat)
    y_host = torch.empty_like(y_flat, device="cpu").pin_memory()
    a_flat2, a_views2 = _aligned_views(torch, [(c.M, c.K) for c in cases], a_flat.dtype, device)
    y_flat2, y_views2 = _aligned_views(torch, [(c.M, c.N) for c in cases], y_flat.dtype, device)
    a_bufs, y_bufs = (a_flat, a_flat2), (y_flat, y_flat2)
    a_sets, y_sets = (a_views, a_views2), (y_views, y_views2)
    io_in, io_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    e2e_graphs = {}
    for b in (0, 1):
        for ri, r in enumerate(rot):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fork = torch.cuda.Event()
                fork.record(stream)
                io_in.wait_event(fork)
                io_out.wait_event(fork)
                with torch.cuda.stream(io_in):
                    a_bufs[1 - b].copy_(a_host, non_blocking=True)   # the next step's input
                with torch.cuda.stream(io_out):
                    y_host.copy_(y_bufs[1 - b], non_blocking=True)   # the previous step's result
                join_in, join_out = torch.cuda.Event(), torch.cuda.Event()
                join_in.record(io_in)
                join_out.record(io_out)
                for c, A, Y in zip(cases, a_sets[b], y_sets[b]):
                    w4.gemm(A, r[c.key], out=Y, workspace=r["workspace"], static_weights=True,
                            **GEMM_KW)
                stream.wait_event(join_in)
                stream.wait_event(join_out)
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
    del e2e_graphs

    value = world * rate(unit, step_bytes, step_flops, secs / args.steps)
    e2e_value = world * rate(unit, step_bytes, step_flops, e2e_secs / args.steps)
    # one kernel per GEMM (W4A8: the activation quantization too)
    launches = len(cases) * args.steps * (2 if GEMM_KW.get("a8") else 1)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.act,
        "data": "synthetic",
        "config": {**workload_config(wl),
                   "activations": args.act,
                   "static_weights": True,
                   "l2": (f"inputs larger than L2: {len(rot)} rotating copies of the packed "
                          f"weights, {len(rot) * packed_bytes / 2**20:.0f} MiB")},
        "tflops": world * step_flops * args.steps / secs / 1e12,
        "hbm_gbs": world * step_bytes * args.steps / secs / 1e9,
        "step_ms_quantiles": {"p10": step_ms[len(step_ms) // 10], "p50": step_ms[len(step_ms) // 2],
                              "p90": step_ms[(9 * len(step_ms)) // 10]},
        "roofline_frac_step": step_roof_us * 1e-6 * args.steps / secs,
        "roofline": roofline,
        "roofline_by_bound": groups,
        "e2e": {"value": e2e_value, "unit": unit,
                "copies": "double-buffered on one stream per direction: step i overlaps the "
                          "input copy of step i+1 and the result copy of step i-1",
                "h2d_bytes_per_step": sum(2 * c.M * c.K for c in cases),
                "d2h_bytes_per_step": sum(2 * c.M * c.N for c in cases)},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if not args.no_by_m:
        # per M (outside the timed region): a graph of 20 launches per case
        times = per_case_times(torch, w4, cases, rot, a_views, y_views, stream)
        by_m = {}
        for c, t in zip(cases, times):
            d = by_m.setdefault(c.M, {"bytes": 0, "flops": 0, "s": 0.0, "roof_us": 0.0})
            d["bytes"] += alg_bytes(c.M, c.K, c.N, c.group)
            d["flops"] += flops(c.M, c.K, c.N)
            d["s"] += t
            d["roof_us"] += roofline_us(c.M, c.K, c.N, c.group, pk)[0]
        line["by_m"] = {str(m): {"TFLOP/s": d["flops"] / d["s"] / 1e12, "GB/s": d["bytes"] / d["s"] / 1e9,
                                 "us": 1e6 * d["s"], "roofline_frac": d["roof_us"] * 1e-6 / d["s"]}
                        for m, d in sorted(by_m.items())}
        line["by_m_how"] = ("per case: a CUDA graph of 20 launches over the rotating weight "
                            "copies, outside the timed region; summed over the layers and groups")
        if args.sweep:
            with open(args.sweep, "a") as f:
                for c, t in zip(cases, times):
                    roof, bound = roofline_us(c.M, c.K, c.N, c.group, pk)
                    path, parts_n = w4.plan(c.M, c.N, c.K, c.group)
                    f.write(json.dumps({
                        "workload": wl.name, "act": args.act, "layer": c.layer, "M": c.M,
                        "K": c.K, "N": c.N, "group": c.group, "path": path, "parts": parts_n,
                        "us": 1e6 * t, "GBps": alg_bytes(c.M, c.K, c.N, c.group) / t / 1e9,
                        "TFLOPs": flops(c.M, c.K, c.N) / t / 1e12, "roofline_us": roof,
                        "bound": bound, "frac": roof / (1e6 * t)}) + "\n")
                for c, t in silu_mul_times(torch, w4, cases, rot, a_views, stream):
                    # the fused layer writes half the columns
                    nbytes = alg_bytes(c.M, c.K, c.N, c.group) - c.M * c.N
                    f.write(json.dumps({
                        "workload": wl.name, "act": args.act, "layer": "gate_up+silu_mul",
                        "M": c.M, "K": c.K, "N": c.N, "group": c.group, "us": 1e6 * t,
                        "GBps": nbytes / t / 1e9, "TFLOPs": flops(c.M, c.K, c.N) / t / 1e12}) + "\n")
    # host cost of one eager call of the smallest GEMM (outside graphs)
    small = min(range(len(cases)), key=lambda i: (cases[i].M, cases[i].N * cases[i].K))
    line["host_us_per_call"] = {
        **host_call_us(torch, w4, cases[small], rot[0], a_views[small], y_views[small], stream),
        "case": f"{cases[small].layer} M={cases[small].M} K={cases[small].K} N={cases[small].N} "
                f"group={cases[small].group}",
        "how": "200 eager calls, host time to enqueue (no synchronization inside the loop)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, unit)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=4, help="workload index (0..4)")
    ap.add_argument("--copies", type=int, default=None, help="weight copies for L2 rotation")
    ap.add_argument("--sweep", default=None, help="append per-case timings (JSONL) here")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-by-m", action="store_true", help="skip the per-M table")
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
