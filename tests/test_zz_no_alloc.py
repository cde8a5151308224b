"""w4a16_gemm_noalloc: the entry point for callers that cannot allocate.

Some callers may not allocate device memory once they run (a fixed memory
budget, a plugin without access to its host's allocator). For them the
library offers a decode-path GEMM that takes no workspace and uses a device
array inside the library instead. This file checks, through the C ABI, that
two calls in a row give the same results as the regular entry point: within
the parity tolerance 2^-9 * sum|a*w| + 1e-3 per element, and bit for bit
(both run the same kernel with the same CTA count and summation order). It is collected
last so that a failure here never hides the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits, prepare

pytestmark = pytest.mark.gpu


def _noalloc(lib, A, pw, Y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.w4a16_gemm_noalloc(A.data_ptr(), pw.Wq.data_ptr(), pw.Sp.data_ptr(),
                                  pw.Zp.data_ptr(), A.shape[0], pw.N, pw.K, pw.group,
                                  Y.data_ptr(), stream)


@pytest.mark.parametrize("M,K,N,group", [(1, 4096, 4096, 128), (16, 2048, 1040, 128),
                                         (5, 1024, 400, 1024), (21, 1024, 272, 64)])
def test_noalloc_matches_regular_entry_point_on_two_calls(M, K, N, group):
    lib = w4.lib()
    W = synthetic.small_weights(K, N, seed=70 + M)
    (q, s, z), pw = prepare(W, group)
    _, mag = oracle.reference(synthetic.small_activations(M, K, seed=70 + M), q, s, z, group)
    bound = 2.0 ** -9 * mag + 1e-3
    for call in range(2):  # the second call runs on the scratch the first one left behind
        A = synthetic.small_activations(M, K, seed=70 + M)
        if call == 1:
            A = (A.astype(np.float32) * -0.5).astype(np.float16)  # new inputs, same magnitudes
            _, mag = oracle.reference(A, q, s, z, group)
            bound = 2.0 ** -9 * mag + 1e-3
        Ad = cuda(A)
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        rc = _noalloc(lib, Ad, pw, Y)
        assert rc == 0, lib.w4a16_last_error().decode()
        ref = w4.gemm(Ad, pw, path="decode-streamk")
        w4.device_status()
        diff = np.abs(oracle.from_half(half_bits(Y)) - oracle.from_half(half_bits(ref)))
        assert np.all(diff <= bound), f"call {call}: max diff/bound {np.max(diff / bound)}"
        # same kernel, same CTA count, same fixed summation order: the same bits
        assert np.array_equal(half_bits(Y), half_bits(ref)), f"call {call}: not bitwise equal"


def test_noalloc_rejects_a_stream_of_another_device():
    if torch.cuda.device_count() < 2:
        pytest.skip("one device: no stream of another device to pass")
    lib = w4.lib()
    pw = prepare(synthetic.small_weights(128, 32, seed=1), 128)[1]
    A = torch.zeros((1, 128), dtype=torch.float16, device="cuda")
    Y = torch.empty((1, 32), dtype=torch.float16, device="cuda")
    other = torch.cuda.Stream(device=1)
    assert lib.w4a16_gemm_noalloc(A.data_ptr(), pw.Wq.data_ptr(), pw.Sp.data_ptr(),
                                  pw.Zp.data_ptr(), 1, 32, 128, 128, Y.data_ptr(),
                                  ctypes.c_void_p(other.cuda_stream)) == -1


def test_noalloc_rejects_bad_arguments():
    lib = w4.lib()
    pw = prepare(synthetic.small_weights(128, 32, seed=1), 128)[1]
    A = torch.zeros((1, 128), dtype=torch.float16, device="cuda")
    Y = torch.empty((1, 32), dtype=torch.float16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.w4a16_gemm_noalloc(None, pw.Wq.data_ptr(), pw.Sp.data_ptr(), pw.Zp.data_ptr(),
                                  1, 32, 128, 128, Y.data_ptr(), stream) == -1
    assert lib.w4a16_gemm_noalloc(A.data_ptr(), pw.Wq.data_ptr(), pw.Sp.data_ptr(),
                                  pw.Zp.data_ptr(), 1, 40, 128, 128, Y.data_ptr(), stream) == -2
    assert lib.w4a16_last_error()
