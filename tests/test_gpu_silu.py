"""Fused gate/up epilogue parity (W4A16_SILU_MUL): CUDA library vs CPU oracle.

The weight's N columns are [gate | up] and the library returns
Y [M, N/2] = silu(gate) * up (lmdeploy issue #2274 "[Feature] support
qqq(w4a8) for lmdeploy", section "Modification": gate and up fused into one
weight, SiLU fused into the GEMM). The oracle forms the same from its fp64
product and propagates the GEMM's per-element bound through silu and the
product (oracle.silu_mul), so each element is checked against its own bound.
The resident decode variant fuses the epilogue into the GEMM kernel; the
stream-K variant and the tensor-core path run it as a second kernel over a
product kept in the workspace. Every path is forced on every case it takes.
"""
import numpy as np
import pytest

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, guarded_output, check_guard, half_bits, prepare

pytestmark = pytest.mark.gpu


def run_silu(M, K, N, group, seed, path, parts=0, repeat=2):
    W = synthetic.small_weights(K, N, seed)
    A = synthetic.small_activations(M, K, seed)
    (q, s, z), pw = prepare(W, group)
    Ad = cuda(A)
    need = w4.workspace_size(M, N, K, group, path, parts, silu_mul=True)
    ws = w4.new_workspace(need) if need else None
    outs = []
    for _ in range(repeat):
        full, Y, pad = guarded_output(M, N // 2)
        try:
            w4.gemm(Ad, pw, out=Y, path=path, parts=parts, workspace=ws, silu_mul=True)
        except w4.W4A16Error as e:
            if path == "decode-resident" and e.code == -2:
                pytest.skip("activations do not fit the resident variant")
            raise
        w4.device_status()
        check_guard(full, M, N // 2, pad)
        outs.append(half_bits(Y).copy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "repeated call is not bitwise identical"
    y, mag = oracle.reference(A, q, s, z, group)
    ref, bound = oracle.silu_mul(y, mag)
    ratio, idx = oracle.check_bound(outs[0], ref, bound)
    h = N // 2
    assert ratio <= 1.0, (f"max err/bound {ratio:.3f} at (m={idx // h}, n={idx % h}): got "
                          f"{oracle.from_half(outs[0].reshape(-1)[idx])}, want {ref.reshape(-1)[idx]}")
    return outs[0]


DECODE_CASES = [
    # M, K, N, group, CTAs (0: automatic)
    (1, 256, 32, 64, 1),        # one pair of strips
    (1, 512, 64, 128, 0),
    (2, 512, 64, 128, 2),       # one pair per CTA
    (4, 1024, 352, 128, 3),     # 11 pairs over 3 CTAs: a ragged split
    (8, 4096, 1024, 128, 0),
    (9, 640, 288, 640, 5),      # one group per column, two token octets
    (16, 4096, 2048, 128, 0),
    (3, 11008, 256, 128, 0),    # 16 warps, about 90 KiB of staged rows
    (12, 2048, 1056, 2048, 7),
    # more strips per CTA than warps, scale records too small to hold a
    # finished strip: finished strips in a region of their own
    (1, 512, 640, 128, 1),
    (6, 1024, 1280, 128, 2),
    # more strips per CTA than warps, finished strips over their scale records
    (2, 2048, 1024, 128, 2),
    (10, 4096, 2048, 128, 3),
    # 16 rows of K = 5120 over 864 pairs: fits only with the strips over the rows
    (16, 5120, 27648, 128, 0),
]


@pytest.mark.parametrize("path", ["decode-resident", "decode-streamk", "decode"])
@pytest.mark.parametrize("M,K,N,group,parts", DECODE_CASES)
def test_decode_silu_mul(M, K, N, group, parts, path):
    run_silu(M, K, N, group, 7 * M + N, path, parts)


@pytest.mark.parametrize("M,K,N,group,parts", [
    (20, 1024, 320, 128, 0),    # decode path forced above 16 rows: two launches
    (33, 512, 96, 128, 0),
])
def test_decode_silu_mul_many_rows(M, K, N, group, parts):
    run_silu(M, K, N, group, M + N, "decode", parts)


@pytest.mark.parametrize("M,K,N,group,parts", [
    (64, 1024, 512, 128, 0),
    (200, 512, 352, 128, 0),    # ragged token tile, 22 strips
    (33, 4096, 1024, 128, 4),   # K split through the workspace, then the epilogue
    (130, 1024, 2080, 1024, 0),
])
def test_tensor_silu_mul(M, K, N, group, parts):
    run_silu(M, K, N, group, M * 3 + N, "tensor", parts)


def test_shared_workspace_stays_usable():
    """A launch without a K split keeps its product clear of the workspace's
    flag/counter area, so that a later K-split launch on the same workspace
    finds its counters zero."""
    M, K, N, g = 64, 2048, 512, 128
    W = synthetic.small_weights(K, N, 11)
    A = synthetic.small_activations(M, K, 11)
    (q, s, z), pw = prepare(W, g)
    y, mag = oracle.reference(A, q, s, z, g)
    ref, bound = oracle.silu_mul(y, mag)
    ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g, "tensor", p, silu_mul=True)
                              for p in (1, 4)))
    for parts, fused in ((1, True), (4, False), (4, True), (1, True), (4, False)):
        Y = w4.gemm(cuda(A), pw, path="tensor", parts=parts, workspace=ws, silu_mul=fused)
        w4.device_status()
        if fused:
            ratio, _ = oracle.check_bound(half_bits(Y), ref, bound)
        else:
            ratio, _ = oracle.check(half_bits(Y), y, mag)
        assert ratio <= 1.0, (parts, fused, ratio)


def test_odd_strip_count_is_rejected():
    pw = w4.quantize_pack(cuda(synthetic.small_weights(256, 48, 1)), 128)
    A = cuda(synthetic.small_activations(1, 256, 1))
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemm(A, pw, silu_mul=True)
    assert e.value.code == -2


SAMPLED_PAIRS = 16
GATE_UP = [(cfg, K, N, g, sorted({M for (l, M, k, n, gg) in synthetic.workload(cfg).cases()
                                  if l == "gate_up" and (k, n, gg) == (K, N, g)}))
           for cfg, K, N, g in [(1, 4096, 22016, 128), (2, 5120, 27648, 128), (3, 4096, 22016, 128)]]


@pytest.mark.parametrize("cfg,K,N,g,ms", GATE_UP, ids=[f"cfg{c[0]}-gate_up" for c in GATE_UP])
def test_full_size_gate_up(cfg, K, N, g, ms):
    """The workloads' gate_up layers at full size, in the automatic path with
    static weights and one shared workspace, on sampled output columns (both
    halves of each sampled column computed by the oracle over all of K)."""
    W = synthetic.weights(cfg, K, N)
    pw = w4.quantize_pack(cuda(W), g)
    h = N // 2
    cols = synthetic.sample_indices(h, SAMPLED_PAIRS, seed=3, salt=N + cfg)
    both = np.concatenate([cols, cols + h])
    q, s, z = oracle.quantize(np.ascontiguousarray(W[:, both]), g)
    del W
    ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g, silu_mul=True) for M in ms))
    wl = synthetic.workload(cfg)
    for M in ms:
        A = synthetic.activations(cfg, M, K, N, outliers=wl.outliers)
        Y = w4.gemm(cuda(A), pw, workspace=ws, static_weights=True, silu_mul=True)
        w4.device_status()
        got = np.ascontiguousarray(half_bits(Y)[:, cols])
        y, mag = oracle.reference(A, q, s, z, g)
        ref, bound = oracle.silu_mul(y, mag)
        ratio, idx = oracle.check_bound(got, ref, bound)
        assert ratio <= 1.0, (f"{wl.name} gate_up M={M}: max err/bound {ratio:.3f} at row "
                              f"{idx // len(cols)}, column {cols[idx % len(cols)]}")
