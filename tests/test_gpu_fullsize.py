"""Full-size parity: every case of the five workloads at its full shape, in
the launch configuration bench.py times (automatic path and grid, static
weights, one shared workspace), against the oracle on
  - all N columns of 16 seeded rows (every rows when M <= 16), so that every
    column tile, K-split slot and the last, ragged tile are checked, and
  - all M rows of 256 seeded columns.
The oracle quantizes the whole weight itself from the same seeded fp32
values; nothing it uses comes from the GPU. The worst err/bound ratio of every
case is recorded (see conftest.py: printed at the end of the session and
written as JSON to the file W4A16_MARGINS_FILE names, if set)."""
import numpy as np
import pytest

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, half_bits

pytestmark = pytest.mark.gpu

SAMPLED_COLUMNS = 256
SAMPLED_ROWS = 16


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
def test_full_size_case(key, ms, margins):
    cfg, layer, K, N, g = key
    wl = synthetic.workload(cfg)
    W = synthetic.weights(cfg, K, N)
    pw = w4.quantize_pack(cuda(W), g)
    q, s, z = oracle.quantize(W, g)
    del W
    deq = oracle.dequantize(q, s, z, g)
    del q
    cols = synthetic.sample_indices(N, SAMPLED_COLUMNS, seed=1, salt=N + 7 * cfg)
    deq_cols = np.ascontiguousarray(deq[:, cols])
    ws = w4.new_workspace(max(w4.workspace_size(M, N, K, g) for M in ms))
    for M in ms:
        A = synthetic.activations(cfg, M, K, N, outliers=wl.outliers)
        Y = w4.gemm(cuda(A), pw, workspace=ws, static_weights=True)
        w4.device_status()
        bits = half_bits(Y)
        path, parts = w4.plan(M, N, K, g)
        where = f"{wl.name} {layer} M={M} g={g} ({path}, {parts})"
        # all M rows of the sampled columns
        y, mag = oracle.matmul(A, deq_cols)
        ratio_c, idx = oracle.check(np.ascontiguousarray(bits[:, cols]), y, mag)
        assert ratio_c <= 1.0, (f"{where}: max err/bound {ratio_c:.3f} at row "
                                f"{idx // len(cols)}, column {cols[idx % len(cols)]}")
        # every column of the sampled rows
        rows = (np.arange(M) if M <= SAMPLED_ROWS
                else synthetic.sample_indices(M, SAMPLED_ROWS, seed=2, salt=M + N))
        y, mag = oracle.matmul(np.ascontiguousarray(A[rows]), deq)
        ratio_r, idx = oracle.check(np.ascontiguousarray(bits[rows]), y, mag)
        assert ratio_r <= 1.0, (f"{where}: max err/bound {ratio_r:.3f} at row "
                                f"{rows[idx // N]}, column {idx % N}")
        margins.append({"test": "full_size", "workload": wl.name, "layer": layer, "M": M,
                        "K": K, "N": N, "group": g, "path": path, "parts": parts,
                        "max_err_over_bound": max(ratio_c, ratio_r)})
