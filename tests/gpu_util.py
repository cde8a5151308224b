"""Helpers shared by the GPU parity tests (CUDA library vs CPU oracle)."""
import numpy as np
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic

# worst err/bound ratio of each parity case: dicts with "test", "path" and
# "max_err_over_bound" (and the case's shape), reported by conftest.py
MARGINS = []


def cuda(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def half_bits(t: torch.Tensor) -> np.ndarray:
    return host(t).view(np.uint16)


def prepare(W: np.ndarray, group: int):
    """Quantize on both sides, check the codes agree bit for bit, pack on the GPU."""
    q, s, z = oracle.quantize(W, group)
    qg, sg, zg = w4.quantize(cuda(W), group)
    assert np.array_equal(host(qg), q), "quantized codes differ from the oracle"
    assert np.array_equal(half_bits(sg), s), "scales differ from the oracle"
    assert np.array_equal(host(zg), z), "zero points differ from the oracle"
    return (q, s, z), w4.pack(qg, sg, zg, group)


def guarded_output(M: int, N: int, pad: int = 64):
    """Y inside a sentinel-filled buffer; returns (full, view, pad)."""
    full = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device="cuda")
    full.view(torch.int16)[:] = 0x7E5A   # a NaN payload no kernel writes
    return full, full[pad:pad + M * N].view(M, N), pad


def check_guard(full: torch.Tensor, M: int, N: int, pad: int):
    bits = host(full.view(torch.int16)).view(np.uint16)
    assert np.all(bits[:pad] == 0x7E5A), "write before Y"
    assert np.all(bits[pad + M * N:] == 0x7E5A), "write after Y"


def run_and_check(M, K, N, group, seed, path="auto", parts=0, outliers=False, repeat=2):
    W = synthetic.small_weights(K, N, seed)
    A = synthetic.small_activations(M, K, seed, outliers=outliers)
    (q, s, z), pw = prepare(W, group)
    Ad = cuda(A)
    outs = []
    for _ in range(repeat):
        full, Y, pad = guarded_output(M, N)
        w4.gemm(Ad, pw, out=Y, path=path, parts=parts)
        w4.device_status()
        check_guard(full, M, N, pad)
        outs.append(half_bits(Y).copy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "repeated call is not bitwise identical"
    y, mag = oracle.reference(A, q, s, z, group)
    ratio, idx = oracle.check(outs[0], y, mag)
    MARGINS.append({"test": "small", "path": path if path != "auto" else w4.plan(M, N, K, group)[0],
                    "M": M, "K": K, "N": N, "group": group, "parts": parts,
                    "max_err_over_bound": float(ratio)})
    assert ratio <= 1.0, (f"max err/bound {ratio:.3f} at (m={idx // N}, n={idx % N}): "
                          f"got {oracle.from_half(outs[0].reshape(-1)[idx])}, want {y.reshape(-1)[idx]}")
    return ratio
