"""Full-size parity: every case of the five workloads at its full shape, in
the launch configuration bench.py times (automatic path and grid, static
weights, one shared workspace), checked on a seeded sample of output columns
that the oracle computes in full (every row, all of K).

The GPU quantizes and packs the whole weight; the oracle quantizes the
sampled columns only (quantization is per column and group, and the GPU
quantizer is bit-exact with the oracle's, see test_gpu_prep.py)."""
import numpy as np
import pytest

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits

pytestmark = pytest.mark.gpu

SAMPLED_COLUMNS = 24


def _layers():
    """Each distinct (workload, layer, K, N, group) once, with all its M."""
    out = {}
    for cfg in range(5):
        for (layer, M, K, N, g) in synthetic.workload(cfg).cases():
            out.setdefault((cfg, layer, K, N, g), []).append(M)
    return sorted(out.items())


LAYERS = _layers()


@pytest.mark.parametrize("key,ms", LAYERS,
                         ids=[f"cfg{k[0]}-{k[1]}-K{k[2]}-N{k[3]}-g{k[4]}" for k, _ in LAYERS])
def test_full_size_case(key, ms):
    cfg, layer, K, N, g = key
    wl = synthetic.workload(cfg)
    W = synthetic.weights(cfg, K, N)
    pw = w4.quantize_pack(cuda(W), g)
    cols = synthetic.sample_indices(N, SAMPLED_COLUMNS, seed=1, salt=N + 7 * cfg)
    q, s, z = oracle.quantize(np.ascontiguousarray(W[:, cols]), g)
    del W
    ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g) for M in ms))
    for M in ms:
        A = synthetic.activations(cfg, M, K, N, outliers=wl.outliers)
        Y = w4.gemm(cuda(A), pw, workspace=ws, static_weights=True)
        w4.device_status()
        got = np.ascontiguousarray(half_bits(Y)[:, cols])
        y, mag = oracle.reference(A, q, s, z, g)
        ratio, idx = oracle.check(got, y, mag)
        path, parts = w4.plan(M, N, K, g)
        assert ratio <= 1.0, (f"{wl.name} {layer} M={M} ({path}, {parts}): max err/bound "
                              f"{ratio:.3f} at row {idx // len(cols)}, column {cols[idx % len(cols)]}")
