"""GEMM parity: CUDA library vs CPU oracle, element by element.

Tolerance (per element): |y - y_ref| <= 2^-9 * sum_k |a_k w_kn| + 1e-3, with
y_ref the fp64 product of the same fp16 activations and the same
fp16-dequantized weights. Shapes span several CTAs and ragged tails in N (at
the 16-column granularity of the format), in M and in the K split. The decode
path's two variants (activations resident in shared memory, whole strips per
CTA; stream-K with streamed activations) are each forced on every case the
variant takes.
"""
import numpy as np
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
import oracle
import synthetic
from gpu_util import cuda, guarded_output, check_guard, half_bits, host, prepare, run_and_check

pytestmark = pytest.mark.gpu

VARIANTS = ["decode-resident", "decode-streamk"]


def run_variant(M, K, N, group, seed, path, parts=0, **kw):
    """run_and_check, skipping shapes the resident variant does not take."""
    try:
        return run_and_check(M, K, N, group, seed=seed, path=path, parts=parts, **kw)
    except w4.W4A16Error as e:
        if path == "decode-resident" and e.code == -2:
            pytest.skip("activations do not fit the resident variant")
        raise

DECODE_CASES = [
    # M, K, N, group, persistent CTAs (0: automatic)
    (1, 64, 16, 64, 1),
    (1, 128, 16, 128, 2),
    (3, 256, 48, 128, 0),
    (8, 512, 144, 128, 4),
    (9, 640, 272, 64, 3),
    (16, 1024, 256, 1024, 8),
    (16, 4096, 512, 128, 0),
    (2, 4096, 4096, 128, 0),
    (5, 896, 160, 128, 8),
    (7, 1280, 400, 128, 5),
    (12, 2048, 1040, 2048, 2),
    (4, 11008, 256, 128, 0),
    (8, 11008, 128, 128, 0),   # resident: 16 warps, about 224 KiB of shared memory
    (16, 4096, 1040, 128, 0),  # resident: 16 warps, two token octets
]


@pytest.mark.parametrize("path", VARIANTS)
@pytest.mark.parametrize("M,K,N,group,parts", DECODE_CASES)
def test_decode_path(M, K, N, group, parts, path):
    run_variant(M, K, N, group, M * 1000 + N, path, parts)


@pytest.mark.parametrize("M,K,N,group", [(1, 4096, 1024, 128), (8, 4096, 512, 128),
                                         (9, 2048, 256, 128), (16, 4096, 256, 128),
                                         (3, 11008, 256, 128), (4, 11008, 256, 128),
                                         (8, 11008, 256, 128), (16, 11008, 256, 128)])
def test_decode_path_picks_a_variant(M, K, N, group):
    """The automatic choice runs whichever variant plan() reports."""
    variant, _ = w4.plan(M, N, K, group)
    assert variant in VARIANTS
    run_and_check(M, K, N, group, seed=M + K, path="decode")


@pytest.mark.parametrize("M,K,N,group", [(1, 4096, 1024, 128), (16, 4096, 256, 128),
                                         (17, 256, 64, 128), (33, 384, 80, 128),
                                         (24, 1024, 16384, 128), (32, 512, 16400, 128),
                                         (9, 768, 256, 192)])
def test_auto_path(M, K, N, group):
    # (24 rows of a wide layer: two decode passes; 32 rows: tensor cores;
    # group 192: tensor cores)
    run_and_check(M, K, N, group, seed=M + K + N)


def test_outlier_activation_columns():
    run_and_check(4, 4096, 256, 128, seed=5, outliers=True)


@pytest.mark.parametrize("parts", [1, 2, 3, 7, 11, 12, 13, 25, 47, 48, 1000])
def test_every_cta_count_meets_the_tolerance(parts):
    """Stream-K: one CTA (every block whole), blocks shared unevenly between
    CTAs whose runs start inside them, one group per CTA, clamping to the
    3 x 16 = 48 split granules (groups of 2 atoms)."""
    run_and_check(8, 2048, 272, 128, seed=11, path="decode-streamk", parts=parts)


@pytest.mark.parametrize("M", [1, 8, 9])
@pytest.mark.parametrize("parts", [1, 2, 3, 5, 8, 16, 17, 1000])
def test_every_resident_cta_count_meets_the_tolerance(parts, M):
    """Resident variant: all 17 strips in one CTA (warps sharing strips), 2..3
    strips per CTA (strips split between warps at group boundaries), one
    strip per CTA (every warp a part of one strip), clamping to the strips."""
    run_variant(M, 2048, 272, 128, 11 + M, "decode-resident", parts)


@pytest.mark.parametrize("path", VARIANTS)
@pytest.mark.parametrize("M,K,N,group,parts", [(3, 512, 64, 64, 1), (5, 1024, 144, 256, 3),
                                              (9, 2048, 128, 512, 2), (2, 1536, 32, 1536, 2),
                                              (16, 4096, 160, 1024, 3), (1, 320, 48, 320, 1),
                                              (4, 1600, 400, 1600, 5), (7, 704, 96, 64, 0),
                                              (12, 2048, 96, 2048, 2)])
def test_group_sizes(M, K, N, group, parts, path):
    """Groups of 1, 4, 8 and 16 atoms and per-channel groups of any length
    (short last batches of 1..7 atoms at 320, 704, 1600)."""
    run_variant(M, K, N, group, M + K + group, path, parts)


def test_workspace_is_left_zeroed_and_reusable():
    K, N, group = 1024, 400, 128
    W = synthetic.small_weights(K, N, seed=4)
    (q, s, z), pw = prepare(W, group)
    ws = w4.new_workspace(w4.workspace_size(16, N, K, group, path="decode-streamk", parts=9))
    for M in (1, 5, 16, 3):
        A = synthetic.small_activations(M, K, seed=M)
        Y = w4.gemm(cuda(A), pw, path="decode-streamk", parts=9, workspace=ws)
        w4.device_status()
        y, mag = oracle.reference(A, q, s, z, group)
        assert oracle.check(half_bits(Y), y, mag)[0] <= 1.0
        counters = ws[:32768].view(torch.int32).cpu().numpy()
        assert np.all(counters == 0), "counters must be left at zero"


def test_one_workspace_serves_calls_of_different_shapes():
    """Calls of different N, M and CTA count in turn share one workspace."""
    shapes = [(1, 1024, 2816), (16, 512, 256), (4, 2048, 1024), (1, 1024, 2816), (9, 640, 4096)]
    ws = w4.new_workspace(max(w4.workspace_size(16, N, K, 128, path="decode", parts=c)
                              for (_, K, N) in shapes for c in (300, 0, 37)))
    for i, (M, K, N) in enumerate(shapes):
        W = synthetic.small_weights(K, N, seed=40 + i)
        A = synthetic.small_activations(M, K, seed=40 + i)
        (q, s, z), pw = prepare(W, 128)
        for parts in (300, 0, 37):
            Y = w4.gemm(cuda(A), pw, path="decode", parts=parts, workspace=ws)
            w4.device_status()
            y, mag = oracle.reference(A, q, s, z, 128)
            assert oracle.check(half_bits(Y), y, mag)[0] <= 1.0, (M, K, N, parts)


def test_integer_product_is_exact():
    """s = 1, z = 8 and integer activations: the exact integer result fits fp16."""
    K, N, M, group = 512, 64, 4, 128
    rng = np.random.default_rng(8)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 1.0, np.float16)
    A = rng.integers(-2, 3, (M, K)).astype(np.float16)
    exact = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.abs(exact).max() < 2048
    pw = w4.pack(cuda(q), cuda(s), cuda(z), group)
    for path in VARIANTS:
        for parts in (1, 4, 0):
            Y = w4.gemm(cuda(A), pw, path=path, parts=parts)
            assert np.array_equal(Y.cpu().numpy().astype(np.int64), exact), (path, parts)


def test_zero_rows_is_a_noop():
    pw = prepare(synthetic.small_weights(128, 32, seed=1), 128)[1]
    full, Y, pad = guarded_output(0, 32)
    w4.gemm(torch.empty((0, 128), dtype=torch.float16, device="cuda"), pw, out=Y)
    w4.device_status()
    check_guard(full, 0, 32, pad)


def test_stream_ordering_on_a_side_stream():
    W = synthetic.small_weights(1024, 256, seed=2)
    A = synthetic.small_activations(4, 1024, seed=2)
    (q, s, z), pw = prepare(W, 128)
    side = torch.cuda.Stream()
    Ad = cuda(A)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        Y = w4.gemm(Ad, pw)
    side.synchronize()
    y, mag = oracle.reference(A, q, s, z, 128)
    assert oracle.check(half_bits(Y), y, mag)[0] <= 1.0


@pytest.mark.parametrize("path", VARIANTS)
def test_static_weights_keeps_the_order_of_a_layer_chain(path):
    """With W4A16_STATIC_WEIGHTS the kernel reads its weights while the previous
    kernel drains, but its activations only after that kernel is done: a chain
    of layers fed by each other (and by a plain torch kernel in between) gives
    the same bits as the same calls made one at a time."""
    K = N = 1024
    M = 5
    pws, refs = [], []
    for seed in (21, 22, 23):
        (q, s, z), pw = prepare(synthetic.small_weights(K, N, seed), 128)
        pws.append(pw)
        refs.append((q, s, z))
    A = cuda(synthetic.small_activations(M, K, seed=21))

    def chain(static):
        x = A
        outs = []
        for i, pw in enumerate(pws):
            x = w4.gemm(x, pw, path=path, static_weights=static)
            outs.append(x)
            if i == 0:
                x = x * 0.5      # a kernel of another library between two layers
            if not static:
                torch.cuda.synchronize()
        return outs

    plain = [half_bits(y).copy() for y in chain(False)]
    for _ in range(3):
        fast = chain(True)
        w4.device_status()
        for a, b in zip(plain, fast):
            assert np.array_equal(a, half_bits(b)), "static-weights chain differs"
    # and the first layer against the oracle
    y, mag = oracle.reference(host(A), *refs[0], 128)
    assert oracle.check(plain[0], y, mag)[0] <= 1.0


def _cancelling_weights(K, N, group, c, seed):
    """Every group of every column holds one weight -c and zeros elsewhere:
    max = 0, min = -c, so s = c/15, z = 15 and every zero weight gets the code
    q = z = 15. The result is one product per group, while the decode path's
    group terms s*(sum q a - z sum a) subtract two sums that are each about
    15 * sum|a| over the group."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 31, K, N, group]))
    W = np.zeros((K, N), np.float32)
    for j in range(K // group):
        rows = j * group + rng.integers(0, group, size=N)
        W[rows, np.arange(N)] = -c
    return W


@pytest.mark.parametrize("path", VARIANTS + ["tensor"])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_cancellation_in_the_group_terms(M, path, margins):
    # activations with a large common offset and x20 outlier channels, so that
    # sum a over a group is large and of one sign
    K, N, group = 4096, 256, 128
    W = _cancelling_weights(K, N, group, c=2.0, seed=M)
    (q, s, z), pw = prepare(W, group)
    assert np.all(z == 15) and np.mean(q == 15) > 0.99
    rng = np.random.default_rng(np.random.SeedSequence([M, 32, K]))
    A = rng.standard_normal((M, K)) + 3.0
    A[:, synthetic.outlier_columns(K, rng)] *= 20.0
    A = A.astype(np.float16)
    try:
        Y = w4.gemm(cuda(A), pw, path=path)
    except w4.W4A16Error as e:
        if path == "decode-resident" and e.code == -2:
            pytest.skip("activations do not fit the resident variant")
        raise
    w4.device_status()
    y, mag = oracle.reference(A, q, s, z, group)
    ratio, idx = oracle.check(half_bits(Y), y, mag)
    margins.append({"test": "cancellation", "path": path, "M": M, "K": K, "N": N,
                    "group": group, "max_err_over_bound": float(ratio)})
    assert ratio <= 1.0, f"max err/bound {ratio:.3f} at (m={idx // N}, n={idx % N})"
