"""Run and time single W4A16 GEMMs: one layer shape at a time.

    python -m bit_weight_only_g128_gb300.run_case --case 4096x8192x57344g128 [--case ...]
        [--path auto|decode|tensor|...] [--parts P] [--warmup W] [--iters I] [--bf16]

Each case is MxKxN with an optional group suffix (gK is the per-channel
group; default g128). Its weight is drawn on the device from a seeded
generator (N(0, 0.02)), quantized and packed by the library, and multiplied
by a seeded N(0, 1) activation matrix `warmup + iters` times, launched back
to back with a CUDA event between consecutive launches on the launching
stream; each timed launch's interval is printed with the achieved TFLOP/s and
HBM GB/s (algorithmic bytes; weights in L2 after the first launch when they
fit there). The
cases run one after another and each frees its buffers before the next, so
that a profiler can be pointed at a few launches of one shape (for example
`ncu -k regex:tc_ -s <warm-up launches> -c 1 ...`) without the memory of a
whole workload. With --graph L the case is instead timed as a CUDA graph of
L launches over copies of the weight that together exceed L2, as the bench
times its steps.
"""
from __future__ import annotations

import argparse
import json

import torch

import bit_weight_only_g128_gb300 as w4


def parse_case(text: str):
    shape, _, g = text.partition("g")
    M, K, N = (int(v) for v in shape.split("x"))
    group = K if g.upper() == "K" else int(g or 128)
    return M, K, N, group


def alg_bytes(M, K, N, group):
    G = K // group
    return K * N // 2 + 2 * G * N + G * N // 2 + 2 * M * K + 2 * M * N


L2_BYTES = 129 * 1024 * 1024


def run(M, K, N, group, path="auto", parts=0, warmup=1, iters=3, bf16=False, seed=0, graph=0):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    W = torch.randn((K, N), generator=gen, device=dev, dtype=torch.float32) * 0.02
    pw = w4.quantize_pack(W, group)
    del W
    torch.cuda.empty_cache()   # keep only what the GEMM uses on the device
    dt = torch.bfloat16 if bf16 else torch.float16
    A = torch.randn((M, K), generator=gen, device=dev, dtype=torch.float32).to(dt)
    Y = torch.empty((M, N), dtype=dt, device=dev)
    ws = w4.new_workspace(w4.workspace_size(M, N, K, group, path, parts), dev)
    stream = torch.cuda.current_stream()
    if graph:
        return run_graph(M, K, N, group, path, parts, pw, A, Y, ws, graph)
    # every launch queued back to back, an event between consecutive launches:
    # each interval is one launch's device time (the host never idles the GPU)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(warmup + iters + 1)]
    events[0].record(stream)
    for i in range(warmup + iters):
        w4.gemm(A, pw, out=Y, path=path, parts=parts, workspace=ws, static_weights=True)
        events[i + 1].record(stream)
    events[-1].synchronize()
    times = [events[i].elapsed_time(events[i + 1]) * 1e3 for i in range(warmup, warmup + iters)]
    w4.device_status()
    used_path, used_parts = w4.plan(M, N, K, group)
    us = min(times) if times else float("nan")
    return {"M": M, "K": K, "N": N, "group": group, "path": path,
            "plan": used_path if path == "auto" else path, "parts": parts or used_parts,
            "us": times, "best_us": us, "TFLOPs": 2.0 * M * N * K / us / 1e6,
            "GBps": alg_bytes(M, K, N, group) / us / 1e3}


def run_graph(M, K, N, group, path, parts, pw, A, Y, ws, launches):
    """Mean time of one launch in a CUDA graph of `launches` back-to-back
    launches (static weights, as a model's layers run), rotating over enough
    copies of the packed weight that they do not stay in L2 between uses."""
    copies = max(1, -(-3 * L2_BYTES // pw.nbytes))
    ws_copies = [pw] + [w4.PackedWeight(pw.Wq.clone(), pw.Sp.clone(), pw.Zp.clone(), pw.K, pw.N,
                                        pw.group) for _ in range(copies - 1)]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(launches):
            w4.gemm(A, ws_copies[i % copies], out=Y, path=path, parts=parts, workspace=ws,
                    static_weights=True)
    times = []
    with torch.cuda.stream(stream):
        for rep in range(4):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            g.replay()
            end.record(stream)
            end.synchronize()
            if rep > 0:  # the first replay warms up
                times.append(start.elapsed_time(end) * 1e3 / launches)
    w4.device_status()
    used_path, used_parts = w4.plan(M, N, K, group)
    us = min(times)
    return {"M": M, "K": K, "N": N, "group": group, "path": path,
            "plan": used_path if path == "auto" else path, "parts": parts or used_parts,
            "us": times, "best_us": us, "TFLOPs": 2.0 * M * N * K / us / 1e6,
            "GBps": alg_bytes(M, K, N, group) / us / 1e3, "graph_launches": launches,
            "weight_copies": copies}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--case", action="append", required=True, help="MxKxN[gG|gK]")
    ap.add_argument("--path", default="auto")
    ap.add_argument("--parts", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--bf16", action="store_true")
    ap.add_argument("--graph", type=int, default=0,
                    help="time a CUDA graph of this many launches over L2-rotated weight copies")
    args = ap.parse_args()
    for text in args.case:
        M, K, N, group = parse_case(text)
        res = run(M, K, N, group, args.path, args.parts, args.warmup, args.iters, args.bf16,
                  graph=args.graph)
        print(json.dumps(res), flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
