"""W4A8 (W4A16_ACT_A8): CUDA library vs CPU oracle.

compressed-tensors PR #269, the Arm example: 16-bit activations in, 8-bit
activations inside the operation, 8-bit x 4-bit product, 16-bit out (lmdeploy
issue #2274: W4A8 with online activation quantization). The activation codes
and scales decide integers, so they must equal the oracle's bit for bit; the
product is held to the 16-bit bound of the result's type with the magnitude
sum s_a * sum |a_q (q - z) s|. Every path is forced on every case it takes.
"""
import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, host, prepare

pytestmark = pytest.mark.gpu


def bits16(t: torch.Tensor) -> np.ndarray:
    return host(t.view(torch.int16)).view(np.uint16)


def activations(M, K, seed, bf16=False, outliers=False):
    """(device tensor, exact values as doubles) of seeded 16-bit activations."""
    A = synthetic.small_activations(M, K, seed, outliers=outliers)
    if bf16:
        b = oracle.to_bf16(A.astype(np.float64))
        return cuda(b.view(np.int16)).view(torch.bfloat16), oracle.from_bf16(b)
    return cuda(A), A.astype(np.float64)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("M,K", [(1, 64), (5, 4096), (16, 11008), (37, 1024), (300, 512)])
def test_quantize_act_matches_oracle_bitwise(M, K, bf16):
    Ad, Av = activations(M, K, M + K, bf16, outliers=K >= 1024)
    aq, sa = w4.quantize_act(Ad)
    raq, rsa = oracle.quantize_act(Av)
    assert np.array_equal(host(aq), raq)
    assert np.array_equal(host(sa).view(np.uint32), rsa.view(np.uint32))


def test_quantize_act_special_rows():
    K = 256
    A = np.zeros((4, K), np.float16)
    A[1, 7] = -3.0                                     # one value: -> -127, s = 3/127
    A[2] = np.float16(2.0 ** -14) * np.arange(K)       # tiny values
    A[3] = np.float16(60000.0) * np.sign(np.arange(K) - 100)  # huge values
    aq, sa = w4.quantize_act(cuda(A))
    raq, rsa = oracle.quantize_act(A.astype(np.float64))
    assert np.array_equal(host(aq), raq) and np.array_equal(host(sa), rsa)
    assert np.all(raq[0] == 0) and rsa[0] == 1.0 and raq[1, 7] == -127


@pytest.mark.parametrize("bf16", [False, True])
def test_quantize_act_near_midpoints(bf16):
    """Values whose quotient a / s_a lies on or next to k + 1/2 (where a fast
    reciprocal product and the correctly rounded quotient could round apart):
    the codes must still be the oracle's."""
    rng = np.random.default_rng(12)
    rows = []
    for amax in (127.0, 100.0, 3.0, 0.37, 1e-3, 6e4 if not bf16 else 3e38):
        k = rng.integers(-127, 127, 4096)
        a = (k + 0.5) * (amax / 127.0) * (1 + rng.choice([0, 1, -1, 2, -2], 4096) * 2.0 ** -20)
        a[0] = amax
        rows.append(a)
    A = np.array(rows)
    bits = oracle.to_bf16(A) if bf16 else oracle.to_half(A)
    vals = oracle.from_bf16(bits) if bf16 else oracle.from_half(bits)
    Ad = cuda(bits.view(np.int16)).view(torch.bfloat16 if bf16 else torch.float16)
    aq, sa = w4.quantize_act(Ad)
    raq, rsa = oracle.quantize_act(vals)
    assert np.array_equal(host(sa).view(np.uint32), rsa.view(np.uint32))
    assert np.array_equal(host(aq), raq), int((host(aq) != raq).sum())


def run_a8(M, K, N, group, seed, path, parts=0, bf16=False, silu=False):
    W = synthetic.small_weights(K, N, seed)
    Ad, Av = activations(M, K, seed, bf16)
    (q, s, z), pw = prepare(W, group)
    aq, sa = oracle.quantize_act(Av)
    need = w4.workspace_size(M, N, K, group, path, parts, silu_mul=silu, a8=True)
    ws = w4.new_workspace(need) if need else None
    outs = []
    for _ in range(2):
        try:
            Y = w4.gemm(Ad, pw, path=path, parts=parts, workspace=ws, silu_mul=silu, a8=True)
        except w4.W4A16Error as e:
            if path == "decode-resident" and e.code == -2:
                pytest.skip("activations do not fit the resident variant")
            raise
        w4.device_status()
        outs.append(bits16(Y).copy())
    assert np.array_equal(outs[0], outs[1]), "repeated call is not bitwise identical"
    y, mag = oracle.reference_a8(aq, sa, q, s, z, group)
    if silu:
        ref, bound = (oracle.silu_mul_bf16 if bf16 else oracle.silu_mul)(y, mag)
        ratio, idx = (oracle.check_bound_bf16 if bf16 else oracle.check_bound)(outs[0], ref, bound)
    else:
        ref = y
        ratio, idx = (oracle.check_bf16 if bf16 else oracle.check)(outs[0], y, mag)
    cols = ref.shape[1]
    assert ratio <= 1.0, f"max err/bound {ratio:.3f} at (m={idx // cols}, n={idx % cols})"


CASES = [
    # M, K, N, group, parts, path
    (1, 256, 48, 64, 0, "decode-resident"),
    (3, 512, 144, 128, 4, "decode-resident"),
    (16, 4096, 512, 128, 0, "decode-resident"),
    (12, 2048, 1040, 2048, 2, "decode-resident"),
    (1, 256, 48, 64, 0, "decode-streamk"),
    (9, 640, 272, 64, 3, "decode-streamk"),
    (16, 11008, 256, 128, 0, "decode-streamk"),
    (20, 1024, 320, 128, 0, "decode"),       # two launches of the decode path
    (8, 4096, 1024, 128, 0, "decode"),
    (17, 512, 128, 128, 0, "tensor"),
    (100, 640, 272, 64, 0, "tensor"),
    (33, 4096, 1024, 128, 4, "tensor"),      # K split
    (300, 2048, 256, 2048, 2, "tensor"),
]


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("M,K,N,group,parts,path", CASES)
def test_w4a8_gemm(M, K, N, group, parts, path, bf16):
    run_a8(M, K, N, group, 11 * M + N, path, parts, bf16)


@pytest.mark.parametrize("M,K,N,group,parts,path", [
    (4, 1024, 352, 128, 3, "decode-resident"),
    (8, 2048, 1024, 128, 0, "decode-streamk"),
    (64, 1024, 512, 128, 0, "tensor"),
])
def test_w4a8_silu_mul(M, K, N, group, parts, path):
    run_a8(M, K, N, group, M + 3 * N, path, parts, silu=True)


@pytest.mark.parametrize("cfg,layers", [(1, None), (3, ("gate_up",))])
def test_full_size_w4a8(cfg, layers):
    """The 7B decode workload (every layer, every M) and the 7B prefill
    gate_up layer with W4A8 at full size, automatic path, static weights, one
    shared workspace; sampled columns computed by the oracle over all of K."""
    wl = synthetic.workload(cfg)
    by_layer = {}
    for (layer, M, K, N, g) in wl.cases():
        if layers is None or layer in layers:
            by_layer.setdefault((layer, K, N, g), []).append(M)
    for (layer, K, N, g), ms in sorted(by_layer.items()):
        W = synthetic.weights(cfg, K, N)
        pw = w4.quantize_pack(cuda(W), g)
        cols = synthetic.sample_indices(N, 16, seed=7, salt=N + 5 * cfg)
        q, s, z = oracle.quantize(np.ascontiguousarray(W[:, cols]), g)
        del W
        ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g, a8=True) for M in ms))
        for M in ms:
            A = synthetic.activations(cfg, M, K, N, outliers=wl.outliers)
            Y = w4.gemm(cuda(A), pw, workspace=ws, static_weights=True, a8=True)
            w4.device_status()
            aq, sa = oracle.quantize_act(A.astype(np.float64))
            y, mag = oracle.reference_a8(aq, sa, q, s, z, g)
            ratio, idx = oracle.check(np.ascontiguousarray(bits16(Y)[:, cols]), y, mag)
            assert ratio <= 1.0, (f"{wl.name} {layer} M={M}: max err/bound {ratio:.3f} at row "
                                  f"{idx // len(cols)}, column {cols[idx % len(cols)]}")
