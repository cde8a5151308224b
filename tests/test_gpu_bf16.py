"""bf16 activations (W4A16_BF16): CUDA library vs CPU oracle.

compressed-tensors PR #269 "Some fixes for AWQ": W4A16 keeps the activations
as unquantized 16-bit floats; a reply names an API taking fp32, bf16 or fp16
activations. A and Y are bf16, the quantized weights the same buffers as for
fp16. The oracle's reference is the fp64 product of the bf16 activations and
the bf16-dequantized weights RNE_bf16((q - z) s); the bound per element is
2^-6 sum|a w| + 1e-3 (four units of bf16 rounding). Every path is forced on
every case it takes, with the same shapes as the fp16 tests: several tiles,
ragged strips, ragged token tiles, K splits, every group form.
"""
import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, host, prepare

pytestmark = pytest.mark.gpu


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return host(t.view(torch.int16)).view(np.uint16)


def guarded_bf16(M, N, pad=64):
    full = torch.empty((M * N + 2 * pad,), dtype=torch.bfloat16, device="cuda")
    full.view(torch.int16)[:] = 0x7FA5  # a NaN payload no kernel writes
    return full, full[pad:pad + M * N].view(M, N), pad


def check_guard_bf16(full, M, N, pad):
    bits = bf16_bits(full)
    assert np.all(bits[:pad] == 0x7FA5), "write before Y"
    assert np.all(bits[pad + M * N:] == 0x7FA5), "write after Y"


def activations_bf16(M, K, seed, outliers=False):
    """The fp16 tests' activations (N(0, 1), optional x20 columns) rounded to bf16."""
    A = synthetic.small_activations(M, K, seed, outliers=outliers)
    return oracle.to_bf16(A.astype(np.float64))


def as_bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    return cuda(bits.view(np.int16)).view(torch.bfloat16)


def run_bf16(M, K, N, group, seed, path, parts=0, silu=False, outliers=False, repeat=2):
    W = synthetic.small_weights(K, N, seed)
    Ab = activations_bf16(M, K, seed, outliers)
    (q, s, z), pw = prepare(W, group)
    Ad = as_bf16_tensor(Ab)
    need = w4.workspace_size(M, N, K, group, path, parts, silu_mul=silu)
    ws = w4.new_workspace(need) if need else None
    ncols = N // 2 if silu else N
    outs = []
    for _ in range(repeat):
        full, Y, pad = guarded_bf16(M, ncols)
        try:
            w4.gemm(Ad, pw, out=Y, path=path, parts=parts, workspace=ws, silu_mul=silu)
        except w4.W4A16Error as e:
            if path == "decode-resident" and e.code == -2:
                pytest.skip("activations do not fit the resident variant")
            raise
        w4.device_status()
        check_guard_bf16(full, M, ncols, pad)
        outs.append(bf16_bits(Y).copy())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "repeated call is not bitwise identical"
    y, mag = oracle.reference_bf16(Ab, q, s, z, group)
    if silu:
        ref, bound = oracle.silu_mul_bf16(y, mag)
        ratio, idx = oracle.check_bound_bf16(outs[0], ref, bound)
    else:
        ref = y
        ratio, idx = oracle.check_bf16(outs[0], y, mag)
    assert ratio <= 1.0, (f"max err/bound {ratio:.3f} at (m={idx // ncols}, n={idx % ncols}): got "
                          f"{oracle.from_bf16(outs[0].reshape(-1)[idx])}, want {ref.reshape(-1)[idx]}")
    return ratio


@pytest.mark.parametrize("K,N,group", [(256, 48, 64), (512, 96, 128), (1024, 160, 256),
                                       (640, 64, 640), (4096, 32, 4096)])
def test_dequantize_bf16_matches_oracle_bitwise(K, N, group):
    (q, s, z), pw = prepare(synthetic.small_weights(K, N, seed=K + N), group)
    got = bf16_bits(w4.dequantize(pw, dtype=torch.bfloat16))
    assert np.array_equal(got, oracle.dequantize_bf16(q, s, z, group))


DECODE_CASES = [
    # M, K, N, group, CTAs (0: automatic)
    (1, 64, 16, 64, 1),
    (1, 128, 16, 128, 2),
    (3, 256, 48, 128, 0),
    (8, 512, 144, 128, 4),
    (9, 640, 272, 64, 3),
    (16, 1024, 256, 1024, 8),
    (16, 4096, 512, 128, 0),
    (5, 896, 160, 128, 8),
    (12, 2048, 1040, 2048, 2),
    (4, 11008, 256, 128, 0),
    (16, 4096, 1040, 128, 0),
]


@pytest.mark.parametrize("path", ["decode-resident", "decode-streamk", "decode"])
@pytest.mark.parametrize("M,K,N,group,parts", DECODE_CASES)
def test_decode_bf16(M, K, N, group, parts, path):
    run_bf16(M, K, N, group, 3 * M + N, path, parts)


@pytest.mark.parametrize("M,K,N,group,parts", [
    (17, 512, 128, 128, 0),
    (64, 1024, 512, 128, 0),
    (100, 640, 272, 64, 0),     # ragged token tile and strips
    (200, 512, 352, 128, 0),
    (33, 4096, 1024, 128, 4),   # K split
    (130, 1024, 2080, 1024, 0),
    (300, 2048, 256, 2048, 2),
])
def test_tensor_bf16(M, K, N, group, parts):
    run_bf16(M, K, N, group, M + 5 * N, "tensor", parts)


def test_outlier_columns_bf16():
    run_bf16(8, 4096, 256, 128, 41, "decode", outliers=True)
    run_bf16(96, 4096, 256, 128, 42, "tensor", outliers=True)


@pytest.mark.parametrize("M,K,N,group,parts,path", [
    (1, 512, 64, 128, 0, "decode-resident"),
    (4, 1024, 352, 128, 3, "decode-resident"),
    (10, 4096, 2048, 128, 3, "decode-resident"),
    (6, 1024, 1280, 128, 2, "decode-resident"),
    (8, 2048, 1024, 128, 0, "decode-streamk"),
    (64, 1024, 512, 128, 0, "tensor"),
    (33, 4096, 1024, 128, 4, "tensor"),
])
def test_silu_mul_bf16(M, K, N, group, parts, path):
    run_bf16(M, K, N, group, M * 7 + N, path, parts, silu=True)


def test_integer_product_is_exact_bf16():
    """s = 1, z = 8 and integer activations: every path forms the exact
    integer in fp32 and rounds it once, so Y equals RNE_bf16(exact)."""
    K, N, M, group = 512, 64, 20, 128
    rng = np.random.default_rng(18)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 1.0, np.float16)
    Ai = rng.integers(-2, 3, (M, K))
    want = oracle.to_bf16((Ai @ (q.astype(np.int64) - 8)).astype(np.float64))
    pw = w4.pack(cuda(q), cuda(s), cuda(z), group)
    A = as_bf16_tensor(oracle.to_bf16(Ai.astype(np.float64)))
    for path, rows in (("decode-resident", 16), ("decode-streamk", 16), ("tensor", 20)):
        for parts in (1, 4, 0):
            Y = w4.gemm(A[:rows].contiguous(), pw, path=path, parts=parts)
            w4.device_status()
            assert np.array_equal(bf16_bits(Y), want[:rows]), (path, parts)


def test_bf16_and_fp16_calls_share_weights_and_workspace():
    """One packed weight and one workspace serve fp16 and bf16 calls in turn."""
    M, K, N, g = 12, 2048, 512, 128
    W = synthetic.small_weights(K, N, 30)
    (q, s, z), pw = prepare(W, g)
    A16 = synthetic.small_activations(M, K, 30)
    Ab = oracle.to_bf16(A16.astype(np.float64))
    ws = w4.new_workspace(w4.workspace_size(M, N, K, g, "decode-streamk"))
    y16, m16 = oracle.reference(A16, q, s, z, g)
    yb, mb = oracle.reference_bf16(Ab, q, s, z, g)
    for _ in range(2):
        Y = w4.gemm(cuda(A16), pw, path="decode-streamk", workspace=ws)
        assert Y.dtype == torch.float16
        assert oracle.check(host(Y.view(torch.int16)).view(np.uint16), y16, m16)[0] <= 1.0
        Yb = w4.gemm(as_bf16_tensor(Ab), pw, path="decode-streamk", workspace=ws)
        assert Yb.dtype == torch.bfloat16
        assert oracle.check_bf16(bf16_bits(Yb), yb, mb)[0] <= 1.0
    w4.device_status()


SAMPLED_COLUMNS = 16


@pytest.mark.parametrize("cfg,layers", [(1, None), (3, ("qkv",))])
def test_full_size_bf16(cfg, layers):
    """The 7B decode workload (every layer, every M) and the 7B prefill qkv
    layer in bf16 at full size, automatic path, static weights, one shared
    workspace; sampled columns computed by the oracle over all of K."""
    wl = synthetic.workload(cfg)
    by_layer = {}
    for (layer, M, K, N, g) in wl.cases():
        if layers is None or layer in layers:
            by_layer.setdefault((layer, K, N, g), []).append(M)
    for (layer, K, N, g), ms in sorted(by_layer.items()):
        W = synthetic.weights(cfg, K, N)
        pw = w4.quantize_pack(cuda(W), g)
        cols = synthetic.sample_indices(N, SAMPLED_COLUMNS, seed=5, salt=N + 3 * cfg)
        q, s, z = oracle.quantize(np.ascontiguousarray(W[:, cols]), g)
        del W
        ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g) for M in ms))
        for M in ms:
            Ab = oracle.to_bf16(synthetic.activations(cfg, M, K, N, outliers=wl.outliers)
                                .astype(np.float64))
            Y = w4.gemm(as_bf16_tensor(Ab), pw, workspace=ws, static_weights=True)
            w4.device_status()
            got = np.ascontiguousarray(bf16_bits(Y)[:, cols])
            y, mag = oracle.reference_bf16(Ab, q, s, z, g)
            ratio, idx = oracle.check_bf16(got, y, mag)
            assert ratio <= 1.0, (f"{wl.name} {layer} M={M}: max err/bound {ratio:.3f} at row "
                                  f"{idx // len(cols)}, column {cols[idx % len(cols)]}")
