"""Parity of the tcgen05/TMEM tensor-core path against the CPU oracle.

Same tolerance as the decode path; shapes cover token tiles of 16..256,
ragged M inside a token tile, several 128-column tiles with a ragged last
tile (N a multiple of 16 only), K from one stage (64) to thousands, and
groups 64, 128 and K (per-channel), and both pipeline stage sizes (64 k, and
128 k for 64-token tiles when K and the group are multiples of 128).
"""
import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits, prepare, run_and_check

pytestmark = pytest.mark.gpu

TENSOR_CASES = [
    # M, K, N, group
    (16, 128, 128, 128),
    (32, 64, 128, 64),
    (128, 256, 256, 128),
    (17, 640, 144, 64),
    (100, 1024, 272, 1024),
    (256, 512, 384, 128),
    (300, 768, 512, 256),
    (64, 4096, 1024, 128),
    (513, 1024, 400, 128),
    (1024, 2048, 1280, 128),
    (8, 256, 16, 128),
    (1, 128, 32, 128),
    # 64-token tiles run 128-k stages when K and the group allow it
    (50, 1152, 144, 128),   # nine 128-k stages, ragged M and N tails
    (60, 1024, 256, 64),    # groups of 64: 64-k stages
    (64, 1088, 128, 1088),  # K not a multiple of 128: 64-k stages
]


@pytest.mark.parametrize("M,K,N,group", TENSOR_CASES)
def test_tensor_path(M, K, N, group):
    run_and_check(M, K, N, group, seed=M * 7 + N, path="tensor")


def test_tensor_outliers():
    run_and_check(512, 4096, 512, 128, seed=3, path="tensor", outliers=True)


@pytest.mark.parametrize("M", [16, 32, 48])
def test_decode_and_tensor_agree(M):
    """Both paths within tolerance of the oracle and within twice it of each other."""
    K, N, group = 2048, 256, 128
    W = synthetic.small_weights(K, N, seed=M)
    A = synthetic.small_activations(M, K, seed=M)
    (q, s, z), pw = prepare(W, group)
    y, mag = oracle.reference(A, q, s, z, group)
    Ad = cuda(A)
    Yd = half_bits(w4.gemm(Ad, pw, path="decode"))
    Yt = half_bits(w4.gemm(Ad, pw, path="tensor"))
    w4.device_status()
    assert oracle.check(Yd, y, mag)[0] <= 1.0
    assert oracle.check(Yt, y, mag)[0] <= 1.0
    diff = np.abs(oracle.from_half(Yd) - oracle.from_half(Yt))
    assert np.all(diff <= 2 * (2.0 ** -9 * mag + 1e-3))


def test_integer_product_is_exact_on_tensor_cores():
    K, N, M, group = 512, 128, 64, 128
    rng = np.random.default_rng(8)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 1.0, np.float16)
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    exact = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    pw = w4.pack(cuda(q), cuda(s), cuda(z), group)
    Y = w4.gemm(cuda(A), pw, path="tensor")
    w4.device_status()
    assert np.array_equal(Y.cpu().numpy().astype(np.int64), exact)


@pytest.mark.parametrize("M,K,N,group,parts", [(64, 4096, 256, 128, 4), (100, 2048, 400, 128, 3),
                                               (300, 1024, 144, 1024, 2), (17, 1280, 48, 64, 5),
                                               (64, 5120, 640, 128, 0), (128, 3072, 1024, 256, 0)])
def test_tensor_k_split(M, K, N, group, parts):
    """K split across CTAs with the last-arriving CTA summing the fp32 tiles."""
    run_and_check(M, K, N, group, seed=M + N + parts, path="tensor", parts=parts)


def test_tensor_split_workspace_is_left_zeroed():
    K, N, group = 2048, 256, 128
    (q, s, z), pw = prepare(synthetic.small_weights(K, N, seed=9), group)
    ws = w4.new_workspace(w4.workspace_size(64, N, K, group, path="tensor", parts=4))
    for M in (64, 40, 64):
        A = synthetic.small_activations(M, K, seed=M)
        Y = w4.gemm(cuda(A), pw, path="tensor", parts=4, workspace=ws)
        w4.device_status()
        y, mag = oracle.reference(A, q, s, z, group)
        assert oracle.check(half_bits(Y), y, mag)[0] <= 1.0
        assert int(ws[:32768].view(torch.int32).abs().sum()) == 0


# the two-SM kernel (cta_group::2): pairs of 128-column halves, 128- or
# 256-token tiles split between the two CTAs; ragged pairs (N not a multiple
# of 256, a second CTA with few or no columns), ragged and partly empty token
# halves (M inside the first half of a tile), every ring depth in use
PAIR_CASES = [
    # M, K, N, group
    (1, 64, 16, 64),
    (17, 128, 256, 128),
    (128, 256, 256, 128),
    (129, 512, 512, 128),
    (256, 1024, 384, 128),   # second pair: one CTA with 128 columns, one with none
    (300, 768, 400, 256),    # second token tile: the second CTA's half is empty
    (512, 4096, 1024, 128),
    (700, 2048, 272, 2048),
    (1024, 1088, 512, 64),   # K not a multiple of 128
    (4096, 512, 768, 128),
    # persistent clusters (76 on GB300) taking several tiles each
    (4000, 128, 2000, 128),  # 128 tiles; ragged last token tile and column pair
    (2304, 64, 4096, 64),    # one stage per tile: the accumulator changes hands every stage
    (1500, 192, 3104, 64),   # 78 tiles: two clusters take a second tile; the last pair has 32 columns
    (8192, 128, 4096, 128),  # about seven tiles per cluster
]


@pytest.mark.parametrize("M,K,N,group", PAIR_CASES)
def test_tensor_pair_path(M, K, N, group):
    run_and_check(M, K, N, group, seed=M * 11 + N, path="tensor-pair")


def test_tensor_pair_outliers_and_auto_choice():
    run_and_check(512, 4096, 512, 128, seed=4, path="tensor-pair", outliers=True)
    # the automatic choice: pairs from 256 rows where they make 80 CTAs
    assert w4.plan(512, 512, 4096, 128)[0] == "tensor"
    assert w4.plan(512, 57344, 8192, 128)[0] == "tensor-pair"
    assert w4.plan(4096, 8192, 8192, 128)[0] == "tensor-pair"
    assert w4.plan(256, 8192, 8192, 128)[0] == "tensor"
    run_and_check(4096, 8192, 8192, 128, seed=5, path="auto", outliers=True)


def test_integer_product_is_exact_on_the_pair():
    K, N, M, group = 512, 256, 300, 128
    rng = np.random.default_rng(18)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 1.0, np.float16)
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    exact = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    pw = w4.pack(cuda(q), cuda(s), cuda(z), group)
    Y = w4.gemm(cuda(A), pw, path="tensor-pair")
    w4.device_status()
    assert np.array_equal(Y.cpu().numpy().astype(np.int64), exact)


@pytest.mark.parametrize("M", [256, 512])
def test_one_and_two_sm_kernels_agree(M):
    """Both tensor-core kernels within tolerance of the oracle; with the same
    operands and fp32 accumulation over the same K order they should agree to
    the last bit or within one unit of the result's rounding."""
    K, N, group = 2048, 512, 128
    W = synthetic.small_weights(K, N, seed=M + 1)
    A = synthetic.small_activations(M, K, seed=M + 1)
    (q, s, z), pw = prepare(W, group)
    y, mag = oracle.reference(A, q, s, z, group)
    Ad = cuda(A)
    Y1 = half_bits(w4.gemm(Ad, pw, path="tensor"))
    Y2 = half_bits(w4.gemm(Ad, pw, path="tensor-pair"))
    w4.device_status()
    assert oracle.check(Y1, y, mag)[0] <= 1.0
    assert oracle.check(Y2, y, mag)[0] <= 1.0
    diff = np.abs(oracle.from_half(Y1) - oracle.from_half(Y2))
    assert np.all(diff <= 2 * (2.0 ** -9 * mag + 1e-3))
