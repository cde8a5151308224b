"""Failure detection without a GPU fault: the kernels' bounded waits give up.

w4a16_selftest_wait launches one kernel whose wait can never be satisfied (a
flag that nothing sets, of the stream-K decode fix-up's kind; an mbarrier
that nothing arrives on, of the tensor-core pipeline's kind), using the
kernels' own wait routines and limit (about a second). The wait must give up,
record its bit in the device error word and let the kernel return: the host
then reads W4A16_ERR_DEVICE_CHECK, the word is cleared, and the context keeps
working. Nothing traps, faults or hangs."""
import re
import time

import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits, prepare

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which,bit", [(0, 32), (1, 2)])
def test_bounded_wait_gives_up_and_reports(which, bit):
    w4.device_status()  # nothing pending
    t0 = time.time()
    w4.selftest_wait(which)
    with pytest.raises(w4.W4A16Error) as e:
        w4.device_status()
    elapsed = time.time() - t0
    assert e.value.code == -6
    word = int(re.search(r"0x([0-9a-f]+)", str(e.value)).group(1), 16)
    assert word == bit, str(e.value)
    assert 0.5 < elapsed < 60, elapsed  # the limit is about a second
    w4.device_status()  # the word was cleared
    # the context still works: a GEMM on each path right after
    K, N, g = 512, 64, 128
    (q, s, z), pw = prepare(synthetic.small_weights(K, N, seed=9), g)
    for M, path in ((3, "decode-streamk"), (24, "tensor")):
        A = synthetic.small_activations(M, K, seed=M)
        y, mag = oracle.reference(A, q, s, z, g)
        Y = w4.gemm(cuda(A), pw, path=path)
        w4.device_status()
        assert oracle.check(half_bits(Y), y, mag)[0] <= 1.0
