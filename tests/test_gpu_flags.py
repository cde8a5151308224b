"""Every combination of the GEMM flags (W4A16_BF16, W4A16_SILU_MUL,
W4A16_ACT_A8) on every path, at the smallest shapes the format allows and at
a ragged one, against the oracle; and zero activations, whose product is
exactly zero on every path and flag."""
import itertools

import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, host, prepare

pytestmark = pytest.mark.gpu

PATHS = ["decode-resident", "decode-streamk", "tensor", "tensor-pair"]


def bits16(t):
    return host(t.view(torch.int16)).view(np.uint16)


def expected(A64, q, s, z, group, bf16, silu, a8):
    if a8:
        aq, sa = oracle.quantize_act(A64)
        y, mag = oracle.reference_a8(aq, sa, q, s, z, group)
    elif bf16:
        y, mag = oracle.reference_bf16(oracle.to_bf16(A64), q, s, z, group)
    else:
        y, mag = oracle.reference(A64.astype(np.float16), q, s, z, group)
    if silu:
        return (oracle.silu_mul_bf16 if bf16 else oracle.silu_mul)(y, mag), True
    return (y, mag), False


@pytest.mark.parametrize("bf16,silu,a8", list(itertools.product([False, True], repeat=3)))
@pytest.mark.parametrize("M,K,N,group", [(1, 64, 32, 64), (3, 64, 32, 64), (19, 192, 96, 64),
                                         (40, 640, 160, 640)])
@pytest.mark.parametrize("path", PATHS)
def test_flag_combinations(path, M, K, N, group, bf16, silu, a8):
    if path == "tensor" and M < 17:
        M += 16  # the tensor path is for more than 16 rows
    check_flags(path, M, K, N, group, bf16, silu, a8)


@pytest.mark.parametrize("bf16,silu,a8", list(itertools.product([False, True], repeat=3)))
def test_flag_combinations_persistent_pairs(bf16, silu, a8):
    """The CTA-pair kernel with more tiles than resident clusters (9 token
    tiles x 13 column pairs), so that clusters take several tiles in turn."""
    check_flags("tensor-pair", 2304, 128, 3328, 128, bf16, silu, a8)


def check_flags(path, M, K, N, group, bf16, silu, a8):
    W = synthetic.small_weights(K, N, seed=M + K + N)
    (q, s, z), pw = prepare(W, group)
    A = synthetic.small_activations(M, K, seed=M * K)
    if bf16:
        b = oracle.to_bf16(A.astype(np.float64))
        A64 = oracle.from_bf16(b)
        Ad = cuda(b.view(np.int16)).view(torch.bfloat16)
    else:
        A64 = A.astype(np.float64)
        Ad = cuda(A)
    need = w4.workspace_size(M, N, K, group, path, 0, silu_mul=silu, a8=a8)
    ws = w4.new_workspace(need) if need else None
    try:
        Y = w4.gemm(Ad, pw, path=path, workspace=ws, silu_mul=silu, a8=a8)
    except w4.W4A16Error as e:
        if path == "decode-resident" and e.code == -2:
            pytest.skip("does not fit the resident variant")
        raise
    w4.device_status()
    assert Y.dtype == (torch.bfloat16 if bf16 else torch.float16)
    assert Y.shape == (M, N // 2 if silu else N)
    (ref, b_or_mag), is_bound = expected(A64, q, s, z, group, bf16, silu, a8)
    got = bits16(Y)
    if is_bound:
        ratio, _ = (oracle.check_bound_bf16 if bf16 else oracle.check_bound)(got, ref, b_or_mag)
    else:
        ratio, _ = (oracle.check_bf16 if bf16 else oracle.check)(got, ref, b_or_mag)
    assert ratio <= 1.0, ratio


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bf16,silu,a8", [(False, False, False), (True, False, False),
                                          (False, True, False), (False, False, True)])
def test_zero_activations_give_zero(path, bf16, silu, a8):
    M, K, N, group = (24 if path == "tensor" else 5), 512, 64, 128
    (q, s, z), pw = prepare(synthetic.small_weights(K, N, seed=3), group)
    Ad = torch.zeros((M, K), dtype=torch.bfloat16 if bf16 else torch.float16, device="cuda")
    need = w4.workspace_size(M, N, K, group, path, 0, silu_mul=silu, a8=a8)
    ws = w4.new_workspace(need) if need else None
    Y = w4.gemm(Ad, pw, path=path, workspace=ws, silu_mul=silu, a8=a8)
    w4.device_status()
    assert np.all(bits16(Y) & 0x7FFF == 0), "a zero input gave a nonzero output"
