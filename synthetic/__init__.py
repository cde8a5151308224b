"""Seeded synthetic inputs for the W4A16 group-quantized linear layer.

This module only draws random numbers and builds shapes. It holds none of the
method's arithmetic (no quantization, no dequantization, no matmul), so both
the CPU oracle and the CUDA library may consume what it produces.

Workloads are synthetic stand-ins for the Llama-2 linear layers on which the
pages discuss AWQ-g128 (vLLM PR #1032 "Implement AWQ quantization support for
LLaMA"; lmdeploy issue #2274 "support qqq(w4a8)", Throughput table): no trained
weights and no datasets are used.

Distributions:
  * W: float32 ~ N(0, 0.02), shape [K, N] (input channels x output channels),
    drawn from numpy's PCG64 with SeedSequence([seed, cfg, K, N]).
  * A: N(0, 1) drawn in float64 with SeedSequence([seed, cfg, K, N, M, 1]);
    for the prefill workload, round(0.01*K) distinct K-columns (chosen with
    the same generator, without replacement) are scaled by 20 before the
    conversion to fp16 (outlier channels).
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np

SEED = 0

# (name, K, N) per model family.
LLAMA2_7B = (("qkv", 4096, 12288), ("o_proj", 4096, 4096),
             ("gate_up", 4096, 22016), ("down", 11008, 4096))
LLAMA2_13B = (("qkv", 5120, 15360), ("o_proj", 5120, 5120),
              ("gate_up", 5120, 27648), ("down", 13824, 5120))
LLAMA2_70B = (("qkv", 8192, 10240), ("o_proj", 8192, 8192),
              ("gate_up", 8192, 57344), ("down", 28672, 8192))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One family of single-linear-layer problems."""
    cfg: int
    name: str
    layers: Tuple[Tuple[str, int, int], ...]
    ms: Tuple[int, ...]
    groups: Tuple[str, ...]       # "128" or "K" (per-channel)
    outliers: bool = False

    def cases(self) -> List[Tuple[str, int, int, int, int]]:
        """All (layer, M, K, N, group) combinations, in a fixed order."""
        out = []
        for gname in self.groups:
            for (layer, K, N) in self.layers:
                g = K if gname == "K" else int(gname)
                for M in self.ms:
                    out.append((layer, M, K, N, g))
        return out


WORKLOADS = (
    Workload(0, "single-4096x4096-m1", (("linear", 4096, 4096),), (1,), ("128",)),
    Workload(1, "llama2-7b-decode", LLAMA2_7B, (1, 4, 8, 16), ("128",)),
    Workload(2, "llama2-13b-mid", LLAMA2_13B, (16, 32, 64, 128), ("128",)),
    Workload(3, "llama2-7b-prefill", LLAMA2_7B, (2048, 4096), ("128",), outliers=True),
    Workload(4, "llama2-70b-sweep", LLAMA2_70B, (1, 8, 64, 512, 4096), ("128", "K")),
)


def workload(cfg: int) -> Workload:
    return WORKLOADS[cfg]


def weights(cfg: int, K: int, N: int, seed: int = SEED) -> np.ndarray:
    """W float32 [K, N] ~ N(0, 0.02)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg, K, N]))
    return rng.standard_normal((K, N), dtype=np.float32) * np.float32(0.02)


def outlier_columns(K: int, rng: np.random.Generator) -> np.ndarray:
    """round(0.01*K) distinct column indices of A (outlier input channels)."""
    count = int(round(0.01 * K))
    return np.sort(rng.choice(K, size=count, replace=False))


def activations(cfg: int, M: int, K: int, N: int, outliers: bool = False,
                seed: int = SEED) -> np.ndarray:
    """A fp16 [M, K] ~ N(0, 1), optionally with x20 outlier columns."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, cfg, K, N, M, 1]))
    a = rng.standard_normal((M, K))
    if outliers:
        cols = outlier_columns(K, rng)
        a[:, cols] *= 20.0
    return a.astype(np.float16)


def small_weights(K: int, N: int, seed: int, scale: float = 0.02) -> np.ndarray:
    """W float32 [K, N] for small parity cases (any shape)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7, K, N]))
    return rng.standard_normal((K, N), dtype=np.float32) * np.float32(scale)


def small_activations(M: int, K: int, seed: int, outliers: bool = False) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 8, M, K]))
    a = rng.standard_normal((M, K))
    if outliers and K >= 100:
        a[:, outlier_columns(K, rng)] *= 20.0
    return a.astype(np.float16)


def sample_indices(total: int, count: int, seed: int, salt: int) -> np.ndarray:
    """Seeded sorted sample of distinct indices in [0, total)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 99, salt, total]))
    count = min(count, total)
    return np.sort(rng.choice(total, size=count, replace=False))


def random_codes(K: int, N: int, group: int, seed: int
                 ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Random quantized triple (q u8 [K,N], s fp16 bits [G,N], z u8 [G,N]).

    Used to exercise packing on arbitrary codes: every nibble value 0..15
    occurs, and s is drawn from normal positive fp16 numbers.
    """
    G = K // group
    rng = np.random.default_rng(np.random.SeedSequence([seed, 11, K, N, group]))
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(0, 16, size=(G, N), dtype=np.uint8)
    s = (rng.uniform(2.0 ** -10, 2.0 ** -4, size=(G, N))).astype(np.float16)
    return q, s.view(np.uint16), z


def grid_group_values(K: int, N: int, group: int, seed: int):
    """Ingredients for weights that lie exactly on the int4 grid.

    Returns (q, s16_bits, z) with, in every group and column, one q == 0 and
    one q == 15 at seeded positions, s16 a normal fp16 in [2^-10, 2^-4] and
    z in [0, 15]. The caller forms w = (q - z) * s itself.
    """
    G = K // group
    rng = np.random.default_rng(np.random.SeedSequence([seed, 13, K, N, group]))
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    for j in range(G):
        lo = rng.integers(0, group, size=N)
        hi = (lo + 1 + rng.integers(0, group - 1, size=N)) % group
        q[j * group + lo, np.arange(N)] = 0
        q[j * group + hi, np.arange(N)] = 15
    z = rng.integers(0, 16, size=(G, N), dtype=np.uint8)
    e = rng.integers(-10, -3, size=(G, N))
    mant = rng.integers(0, 1024, size=(G, N))
    s = np.ldexp(1.0 + mant / 1024.0, e).astype(np.float16)
    return q, s.view(np.uint16), z
