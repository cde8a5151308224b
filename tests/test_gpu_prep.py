"""GPU quantize / pack / unpack / dequantize against the CPU oracle, bit for bit."""
import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits, host, prepare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,N,group", [(128, 16, 128), (4096, 512, 128), (1024, 64, 1024),
                                       (640, 48, 64)])
def test_quantize_matches_oracle(K, N, group):
    prepare(synthetic.small_weights(K, N, seed=K + N), group)


def test_quantize_grid_and_degenerate_groups():
    K, N, group = 256, 64, 128
    q, s, z = synthetic.grid_group_values(K, N, group, seed=1)
    w = ((q.astype(np.int64) - np.repeat(z, group, axis=0)) *
         np.repeat(s.view(np.float16).astype(np.float64), group, axis=0)).astype(np.float32)
    w[:, 0] = 0.0                      # constant zero column: the scale floor
    w[:, 1] = 0.375                    # positive constant
    w[:128, 2] = -2.5                  # negative constant in one group
    w[:, 3] = np.linspace(0, 1e-9, K)  # range far below fp16's smallest scale
    w[:, 4] *= 1000.0                  # large magnitudes
    (q2, s2, z2), _ = prepare(w, group)
    assert np.array_equal(q2[:, 5:], q[:, 5:]) and np.array_equal(z2[:, 5:], z[:, 5:])


@pytest.mark.parametrize("K,N,group", [(64, 16, 64), (256, 48, 128), (1024, 272, 256)])
def test_pack_matches_oracle_and_round_trips(K, N, group):
    q, s, z = synthetic.random_codes(K, N, group, seed=K * N)
    Wp, Sp, Zp = oracle.pack(q, z, s, group)
    pw = w4.pack(cuda(q), cuda(s.view(np.float16)), cuda(z), group)
    assert np.array_equal(host(pw.Wq).view(np.uint32), Wp)
    assert np.array_equal(half_bits(pw.Sp), Sp)
    assert np.array_equal(host(pw.Zp).view(np.uint32), Zp)
    q2, s2, z2 = w4.unpack(pw)
    assert np.array_equal(host(q2), q)
    assert np.array_equal(half_bits(s2), s)
    assert np.array_equal(host(z2), z)


def test_dequantize_matches_oracle_bitwise():
    K, N, group = 512, 64, 128
    rng = np.random.default_rng(3)
    q = rng.integers(0, 16, (K, N), dtype=np.uint8)
    z = rng.integers(0, 16, (K // group, N), dtype=np.uint8)
    # scales over the whole positive finite fp16 range, subnormals included
    s = rng.integers(1, 0x7BFF, (K // group, N)).astype(np.uint16)
    s[0, :8] = [1, 2, 3, 0x3FF, 0x400, 0x7BFF, 0x3C00, 0x00A8]
    pw = w4.pack(cuda(q), cuda(s.view(np.float16)), cuda(z), group)
    deq = half_bits(w4.dequantize(pw))
    ref = oracle.dequantize(q, s, z, group)
    assert np.array_equal(deq, ref)
