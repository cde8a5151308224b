"""Pins for the CPU oracle, each against something other than the oracle.

Sources of truth used here: the IEEE binary16 format (numpy's independent
conversion), a hand-worked example (tests/golden), exact rational arithmetic
(fractions), numpy's float64 matmul, closed forms on the int4 grid, and the
layout text of the packed format re-implemented in this file.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# --------------------------------------------------------------- binary16

def test_from_half_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.from_half(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_to_half_matches_numpy_rounding():
    rng = np.random.default_rng(1)
    # random magnitudes over the whole fp16 range, subnormals and overflow
    x = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 17, 20000)),
        rng.uniform(-1e-7, 1e-7, 2000),
        np.array([65504.0, 65519.99, 65520.0, -65520.0, 1e6, 0.0, -0.0,
                  2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26]),
    ])
    # exact midpoints between adjacent halves: ties must go to even
    h = rng.integers(0, 0x7bff, 5000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    x = np.concatenate([x, (lo + hi) / 2, -(lo + hi) / 2])
    ours = oracle.to_half(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------- worked example

def test_worked_example_group_of_8():
    g = _read_golden("quant_group8_worked.txt")
    w = np.array([float(v) for v in g["w"]], np.float32).reshape(8, 1)
    q, s, z = oracle.quantize(w, 8)
    assert s[0, 0] == int(g["s16_bits"][0], 16)
    assert oracle.from_half(s)[0, 0] == float(g["s16"][0])
    assert z[0, 0] == int(g["z"][0])
    assert q[:, 0].tolist() == [int(v) for v in g["q"]]
    deq = oracle.from_half(oracle.dequantize(q, s, z, 8))[:, 0]
    assert deq.tolist() == [float(v) for v in g["deq"]]
    a = np.array([float(v) for v in g["a"]], np.float16).reshape(1, 8)
    y, mag = oracle.reference(a, q, s, z, 8)
    assert y[0, 0] == float(g["y"][0])
    assert mag[0, 0] == float(g["mag"][0])


# --------------------------------------------------------------- quantizer

def _grid_weights(K, N, group, seed):
    q, s, z = synthetic.grid_group_values(K, N, group, seed)
    G = K // group
    s64 = s.view(np.float16).astype(np.float64)
    qi = q.astype(np.int64)
    zi = np.repeat(z.astype(np.int64), group, axis=0)
    w = (qi - zi) * np.repeat(s64, group, axis=0)      # exact: <= 15 bits
    w32 = w.astype(np.float32)
    assert np.array_equal(w32.astype(np.float64), w)
    return w32, q, s, z, G


@pytest.mark.parametrize("K,N,group", [(256, 32, 128), (128, 16, 32), (192, 8, 64),
                                       (256, 24, 256), (64, 5, 8)])
def test_grid_weights_round_trip_exactly(K, N, group):
    w, q, s, z, _ = _grid_weights(K, N, group, seed=K + N + group)
    q2, s2, z2 = oracle.quantize(w, group)
    assert np.array_equal(s2, s)
    assert np.array_equal(z2, z)
    assert np.array_equal(q2, q)
    # (q - z)*s16 is exact in fp32 (at most 15 significant bits); its fp16
    # rounding is what dequantization must return
    deq = oracle.dequantize(q2, s2, z2, group)
    assert np.array_equal(deq, w.astype(np.float16).view(np.uint16))


def test_quantize_error_bound_random_weights():
    K, N, group = 1024, 96, 128
    w = synthetic.small_weights(K, N, seed=3)
    q, s, z = oracle.quantize(w, group)
    G = K // group
    wg = w.reshape(G, group, N)
    mn, mx = wg.min(axis=1), wg.max(axis=1)
    assert np.all(mn <= 0) and np.all(mx >= 0)
    s32 = ((mx - mn) / np.float32(15)).astype(np.float64)
    s16 = oracle.from_half(s)
    assert np.all(np.abs(s16 - s32) <= s32 * 2.0 ** -11)       # one fp16 rounding
    assert np.all((z >= 0) & (z <= 15)) and np.all(q <= 15)
    recon = (q.astype(np.float64).reshape(G, group, N) - z[:, None, :]) * s16[:, None, :]
    err = np.abs(wg - recon)
    bound = 0.5 * s16 + 15 * np.abs(s32 - s16) + 2.0 ** -20 * s16
    assert np.all(err <= bound[:, None, :])
    # the max element of each group maps to q=15 or its neighbour, the min to q=0 or 1
    deq = oracle.from_half(oracle.dequantize(q, s, z, group)).reshape(G, group, N)
    exact = recon
    ulp_half = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -14))) - 11)
    assert np.all(np.abs(deq - exact) <= ulp_half)


def test_groups_are_independent():
    """Quantizing [W1; W2] with group g equals quantizing W1 and W2 alone."""
    w = synthetic.small_weights(384, 40, seed=4)
    q, s, z = oracle.quantize(w, 128)
    for j in range(3):
        qj, sj, zj = oracle.quantize(w[128 * j:128 * (j + 1)], 128)
        assert np.array_equal(q[128 * j:128 * (j + 1)], qj)
        assert np.array_equal(s[j:j + 1], sj)
        assert np.array_equal(z[j:j + 1], zj)


def test_constant_group_uses_floor_scale():
    w = np.zeros((128, 16), np.float32)
    w[:, 3] = 0.25
    w[:, 4] = -0.125
    q, s, z = oracle.quantize(w, 128)
    floor_bits = np.array([1e-5], np.float64).astype(np.float16).view(np.uint16)[0]
    assert np.all(s == floor_bits)
    assert np.all(z[0, [0, 1, 2, 5]] == 0) and np.all(q[:, 0] == 0)
    # a positive constant is clipped at 15*s (z clamps to 0), a negative one at 0*s
    assert np.all(q[:, 3] == 15) and z[0, 3] == 0
    assert np.all(q[:, 4] == 0) and z[0, 4] == 15


# --------------------------------------------------------------- matmul

def _exact_dot(a, b):
    acc = Fraction(0)
    mag = Fraction(0)
    for x, y in zip(a, b):
        p = Fraction(float(x)) * Fraction(float(y))
        acc += p
        mag += abs(p)
    return acc, mag


def test_matmul_brute_force_tiny():
    rng = np.random.default_rng(5)
    for (M, K, N) in [(1, 1, 1), (2, 3, 4), (3, 8, 5), (4, 17, 3)]:
        A = rng.standard_normal((M, K)).astype(np.float16)
        B = (rng.standard_normal((K, N)) * 0.1).astype(np.float16)
        y, mag = oracle.matmul(A, B)
        for m in range(M):
            for n in range(N):
                ex, exm = _exact_dot(A[m], B[:, n])
                assert abs(y[m, n] - float(ex)) <= 1e-13 * float(exm) + 1e-300
                assert abs(mag[m, n] - float(exm)) <= 1e-13 * float(exm)


def test_matmul_matches_numpy_float64():
    A = synthetic.small_activations(5, 300, seed=6)
    B = (np.random.default_rng(7).standard_normal((300, 70)) * 0.02).astype(np.float16)
    y, mag = oracle.matmul(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    refmag = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * refmag.max())
    assert np.allclose(mag, refmag, rtol=1e-12, atol=0)


def test_integer_closed_form():
    """s = 1, z = 8 and small integer activations give an exact integer product."""
    K, N, M, group = 256, 24, 3, 128
    rng = np.random.default_rng(8)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 0x3C00, np.uint16)          # 1.0
    A = rng.integers(-4, 5, (M, K)).astype(np.float16)
    y, _ = oracle.reference(A, q, s, z, group)
    exact = A.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(y, exact.astype(np.float64))


def test_zero_when_codes_equal_zero_points():
    K, N, group = 256, 16, 128
    z = np.random.default_rng(9).integers(0, 16, (K // group, N)).astype(np.uint8)
    q = np.repeat(z, group, axis=0)
    s = np.full(z.shape, 0x2A66, np.uint16)
    A = synthetic.small_activations(4, K, seed=9)
    y, mag = oracle.reference(A, q, s, z, group)
    assert np.all(y == 0) and np.all(mag == 0)


def test_linear_in_activations():
    K, N, group = 256, 32, 128
    w = synthetic.small_weights(K, N, seed=10)
    q, s, z = oracle.quantize(w, group)
    rng = np.random.default_rng(11)
    A1 = rng.integers(-8, 9, (2, K)).astype(np.float16)
    A2 = rng.integers(-8, 9, (2, K)).astype(np.float16)
    y1, m1 = oracle.reference(A1, q, s, z, group)
    y2, m2 = oracle.reference(A2, q, s, z, group)
    y12, _ = oracle.reference((A1.astype(np.float32) + A2).astype(np.float16), q, s, z, group)
    assert np.allclose(y12, y1 + y2, rtol=0, atol=1e-12 * (m1 + m2).max())


def test_check_accepts_rounded_reference_and_rejects_errors():
    K, N, group = 256, 32, 128
    q, s, z = oracle.quantize(synthetic.small_weights(K, N, seed=12), group)
    A = synthetic.small_activations(3, K, seed=12)
    y, mag = oracle.reference(A, q, s, z, group)
    Y = oracle.to_half(y)
    r, _ = oracle.check(Y, y, mag)
    assert r <= 0.5
    bad = Y.copy()
    bad[1, 5] = oracle.to_half(oracle.from_half(bad[1, 5]) + 0.01 * mag[1, 5] + 0.01)
    r, i = oracle.check(bad, y, mag)
    assert r > 1 and i == 1 * N + 5


# --------------------------------------------------------------- packed layout

def _spec_decode(Wp, K, N):
    """Decode q[k][n] from the packed words using the layout text alone."""
    q = np.empty((K, N), np.uint8)
    natoms = K // 64
    for n in range(N):
        j, c = divmod(n, 16)
        g, r = c % 8, c // 8
        for k in range(K):
            a, kk = divmod(k, 64)
            s_, rem = divmod(kk, 32)
            t, e = divmod(rem, 8)
            word = (j * natoms + a) * 128 + 4 * (4 * g + t) + 2 * s_ + r
            p = int(f"{e:03b}"[::-1], 2)      # nibble = 3-bit reversal of e
            q[k, n] = (int(Wp[word]) >> (4 * p)) & 15
    return q


def test_pack_single_nibble_position():
    K, N = 64, 16
    q = np.zeros((K, N), np.uint8)
    q[9, 3] = 0xA          # atom 0, s=0, t=1, e=1 -> nibble 4; g=3, r=0 -> lane 13, i=0
    z = np.zeros((1, N), np.uint8)
    z[0, 11] = 0x7         # column 8 + 3 -> byte 3 (word 0, bits 24..31), high nibble
    s = np.zeros((1, N), np.uint16)
    s[0, 11] = 0x1234
    Wp, Sp, Zp = oracle.pack(q, z, s, 64)
    expect = np.zeros(K * N // 8, np.uint32)
    expect[4 * 13 + 0] = 0xA << 16
    assert np.array_equal(Wp, expect)
    assert Zp.tolist() == [0x7 << 28, 0]
    assert Sp[7] == 0x1234 and np.count_nonzero(Sp) == 1   # column 11 = 8*1 + 3 -> 2*3 + 1


def test_pack_nibble_order_is_the_bit_reversal_of_the_k_offset():
    # one code per k-offset e = 0..7 of word 0 (column 0, k = e): nibble p
    # must hold e = rev3(p), i.e. nibbles 0..7 hold k-offsets 0 4 2 6 1 5 3 7
    K, N = 64, 16
    q = np.zeros((K, N), np.uint8)
    for e in range(8):
        q[e, 0] = e + 8                      # distinct codes 8..15
    Wp, _, _ = oracle.pack(q, np.zeros((1, N), np.uint8), np.zeros((1, N), np.uint16), 64)
    nibbles = [(int(Wp[0]) >> (4 * p)) & 15 for p in range(8)]
    assert nibbles == [8 + e for e in (0, 4, 2, 6, 1, 5, 3, 7)]
    # so the pair masks of the kernels see consecutive k-offsets
    w = int(Wp[0])
    assert (w & 0xF, (w >> 16) & 0xF) == (8, 9)               # k 0, 1
    assert ((w >> 8) & 0xF, (w >> 24) & 0xF) == (10, 11)      # k 2, 3
    assert ((w >> 4) & 0xF, (w >> 20) & 0xF) == (12, 13)      # k 4, 5
    assert ((w >> 12) & 0xF, (w >> 28) & 0xF) == (14, 15)     # k 6, 7


@pytest.mark.parametrize("K,N,group", [(128, 32, 128), (192, 48, 64), (256, 16, 256)])
def test_pack_follows_layout_text_and_round_trips(K, N, group):
    q, s, z = synthetic.random_codes(K, N, group, seed=K + N)
    Wp, Sp, Zp = oracle.pack(q, z, s, group)
    assert np.array_equal(_spec_decode(Wp, K, N), q)
    G = K // group
    for n in range(N):
        j, c = divmod(n, 16)
        for grp in range(G):
            assert Sp[(j * G + grp) * 16 + 2 * (c % 8) + c // 8] == s[grp, n]
            zbytes = Zp.view(np.uint8)   # little-endian bytes of the word array
            byte = int(zbytes[(j * G + grp) * 8 + c % 8])
            assert (byte >> (4 * (c // 8))) & 15 == z[grp, n]
    q2, s2, z2 = oracle.unpack(Wp, Sp, Zp, K, N, group)
    assert np.array_equal(q2, q) and np.array_equal(s2, s) and np.array_equal(z2, z)


# --- fused gate/up epilogue (lmdeploy issue #2274, "Modification": gate and up
# fused into one weight; element-wise SiLU fused around the GEMM) ----------

def test_silu_odd_even_identities():
    """silu(x) - silu(-x) = x and silu(x) + silu(-x) = x tanh(x/2): the first
    pins the sigmoid's symmetry, the second checks against numpy's tanh."""
    for x in np.linspace(-30.0, 30.0, 241):
        a, b = oracle.silu(x), oracle.silu(-x)
        assert abs((a - b) - x) <= 1e-12 * max(1.0, abs(x))
        assert abs((a + b) - x * np.tanh(x / 2)) <= 1e-12 * max(1.0, abs(x))


def test_silu_limits_and_sign():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12          # sigmoid(40) = 1 - 4e-18
    assert abs(oracle.silu(-40.0)) < 1e-15
    xs = np.linspace(-20, 20, 401)
    vals = np.array([oracle.silu(x) for x in xs])
    assert np.all(vals[xs > 0] > 0) and np.all(vals[xs < 0] < 0)
    # the minimum lies between -1.29 and -1.27 (silu'(x) = 0 there) and is about -0.2785
    xf = np.linspace(-2.0, -0.5, 1501)
    vf = np.array([oracle.silu(x) for x in xf])
    i = int(np.argmin(vf))
    assert -1.29 <= xf[i] <= -1.27 and -0.279 < vf[i] < -0.278


def test_silu_mul_pairs_gate_with_up_half():
    rng = np.random.default_rng(3)
    M, H = 3, 5
    gate = rng.normal(size=(M, H))
    up = rng.normal(size=(M, H))
    y = np.concatenate([gate, up], axis=1)
    out, _ = oracle.silu_mul(y, np.abs(y))
    # zero up -> zero out; zero gate -> zero out; doubling up doubles out exactly
    y0 = np.concatenate([gate, np.zeros_like(up)], axis=1)
    assert np.all(oracle.silu_mul(y0, np.abs(y0))[0] == 0)
    y1 = np.concatenate([np.zeros_like(gate), up], axis=1)
    assert np.all(oracle.silu_mul(y1, np.abs(y1))[0] == 0)
    y2 = np.concatenate([gate, 2 * up], axis=1)
    assert np.array_equal(oracle.silu_mul(y2, np.abs(y2))[0], 2 * out)
    # a large gate passes up through almost unscaled: out ~ gate * up
    y3 = np.concatenate([np.full_like(gate, 40.0), up], axis=1)
    assert np.allclose(oracle.silu_mul(y3, np.abs(y3))[0], 40.0 * up, rtol=1e-12, atol=0)
    # column j of out depends on columns j and H + j only
    for j in range(H):
        yj = y.copy()
        yj[:, j] += 1.0
        d = oracle.silu_mul(yj, np.abs(yj))[0] - out
        assert np.all(d[:, [c for c in range(H) if c != j]] == 0) and np.all(d[:, j] != 0)


def test_silu_mul_bound_accepts_rounding_and_rejects_errors():
    rng = np.random.default_rng(4)
    y = rng.normal(size=(4, 64)) * 3
    mag = np.abs(y) * 4
    out, bound = oracle.silu_mul(y, mag)
    h = oracle.to_half(out)
    assert oracle.check_bound(h, out, bound)[0] <= 1.0
    bad = oracle.to_half(out + 3 * bound)
    assert oracle.check_bound(bad, out, bound)[0] > 1.0


# --------------------------------------------------------------- bf16 activations

def _torch():
    return pytest.importorskip("torch")


def test_from_bf16_all_patterns_match_torch():
    torch = _torch()
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.from_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_to_bf16_matches_torch_rounding():
    """Float32 inputs (so no double rounding on torch's side): normal,
    subnormal, huge and exact-tie values, both signs."""
    torch = _torch()
    rng = np.random.default_rng(21)
    xs = [rng.standard_normal(20000).astype(np.float32),
          (rng.standard_normal(2000) * 1e-39).astype(np.float32),     # bf16 subnormals
          rng.uniform(-3.4e38, 3.4e38, 2000).astype(np.float32),       # near overflow
          np.array([3.4028235e38, -3.4028235e38, 1e-45, 0.0, -0.0], np.float32)]
    # exact ties: 1 + (2j + 1) 2^-8 lies halfway between bf16 neighbours
    j = np.arange(128)
    xs.append(((1.0 + (2 * j + 1) * 2.0 ** -8) * np.where(j % 2, 1.0, -4.0)).astype(np.float32))
    x = np.concatenate(xs)
    ours = oracle.to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # the ties went to the even neighbour
    t = oracle.to_bf16(1.0 + 2.0 ** -8)
    assert t == 0x3F80 and oracle.to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82


def test_dequantize_bf16_matches_torch():
    """RNE_bf16((q - z) * s16): the product is exact in float32 (4 x 11
    significant bits), so torch's float32 -> bf16 rounding is the reference."""
    torch = _torch()
    K, N, group = 256, 48, 64
    q, s, z = oracle.quantize(synthetic.small_weights(K, N, seed=22), group)
    deq = oracle.dequantize_bf16(q, s, z, group)
    sf = oracle.from_half(s).astype(np.float32)
    d = (q.astype(np.int32) - np.repeat(z, group, axis=0).astype(np.int32)).astype(np.float32)
    prod = d * np.repeat(sf, group, axis=0)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(deq, ref)
    # and it is the fp16 dequantization rounded again only where bf16 is coarser
    d16 = oracle.from_half(oracle.dequantize(q, s, z, group))
    assert np.all(np.abs(oracle.from_bf16(deq) - d16) <= 2.0 ** -8 * np.abs(d16) + 2.0 ** -11 * np.abs(d16))


def test_matmul_bf16_brute_force_tiny():
    rng = np.random.default_rng(23)
    for (M, K, N) in [(1, 1, 1), (2, 3, 4), (4, 17, 3)]:
        A = oracle.to_bf16(rng.standard_normal((M, K)))
        B = oracle.to_bf16(rng.standard_normal((K, N)) * 0.1)
        y, mag = oracle.matmul_bf16(A, B)
        Av, Bv = oracle.from_bf16(A), oracle.from_bf16(B)
        for m in range(M):
            for n in range(N):
                ex, exm = _exact_dot(Av[m], Bv[:, n])
                assert abs(y[m, n] - float(ex)) <= 1e-13 * float(exm) + 1e-300
                assert abs(mag[m, n] - float(exm)) <= 1e-13 * float(exm)


def test_integer_closed_form_bf16():
    """s = 1, z = 8 and small integer bf16 activations give an exact integer product."""
    K, N, M, group = 256, 24, 3, 128
    rng = np.random.default_rng(24)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 0x3C00, np.uint16)          # fp16 1.0
    Ai = rng.integers(-4, 5, (M, K))
    A = oracle.to_bf16(Ai)
    y, _ = oracle.reference_bf16(A, q, s, z, group)
    assert np.array_equal(y, (Ai @ (q.astype(np.int64) - 8)).astype(np.float64))


def test_check_bf16_pins_its_bound():
    K, N, group = 256, 32, 128
    q, s, z = oracle.quantize(synthetic.small_weights(K, N, seed=25), group)
    A = oracle.to_bf16(synthetic.small_activations(3, K, seed=25).astype(np.float64))
    y, mag = oracle.reference_bf16(A, q, s, z, group)
    Y = oracle.to_bf16(y)
    assert oracle.check_bf16(Y, y, mag)[0] <= 0.25      # one bf16 rounding: at most 2^-9 |y|
    # the bound is 2^-6 mag + 1e-3: a value just inside passes, just outside fails
    b = 2.0 ** -6 * mag[2, 7] + 1e-3
    for f, ok in ((0.98, True), (1.02, False)):
        ref = y.copy()
        ref[2, 7] = oracle.from_bf16(Y[2, 7]) - f * b
        assert (oracle.check_bf16(Y, ref, mag)[0] <= 1.0) == ok


def test_silu_mul_bf16_bound():
    rng = np.random.default_rng(26)
    y = rng.normal(size=(4, 64)) * 3
    mag = np.abs(y) * 4
    out, bound = oracle.silu_mul_bf16(y, mag)
    out16, bound16 = oracle.silu_mul(y, mag)
    assert np.array_equal(out, out16)                   # the same epilogue
    assert np.all(bound > bound16)                      # under a looser product bound
    assert oracle.check_bound_bf16(oracle.to_bf16(out), out, bound)[0] <= 1.0
    assert oracle.check_bound_bf16(oracle.to_bf16(out + 3 * bound), out, bound)[0] > 1.0


# --------------------------------------------------------------- W4A8

def test_quantize_act_grid_rows_are_exact():
    """Rows c * k with integer k in [-127, 127] reaching 127 and c a power of
    two: amax / 127 = c exactly, so the codes are k and the scale is c."""
    rng = np.random.default_rng(31)
    k = rng.integers(-127, 128, (6, 200))
    k[:, 17] = np.where(np.arange(6) % 2, 127, -127)
    c = 2.0 ** np.array([-12, -6, -1, 0, 3, 5])[:, None]
    aq, sa = oracle.quantize_act(k * c)
    assert np.array_equal(aq, k) and np.array_equal(sa.astype(np.float64), c[:, 0])


def test_quantize_act_error_bound_and_invariants():
    A = oracle.from_half(oracle.to_half(synthetic.small_activations(9, 512, seed=32, outliers=True)
                                        .astype(np.float64)))
    aq, sa = oracle.quantize_act(A)
    # each value within half a step (plus the fp32 rounding of the scale)
    err = np.abs(A - sa[:, None].astype(np.float64) * aq)
    assert np.all(err <= 0.5 * sa[:, None] * (1 + 2.0 ** -20))
    # the largest magnitude of each row maps to +-127, and |a_q| <= 127
    i = np.argmax(np.abs(A), axis=1)
    assert np.all(np.abs(aq[np.arange(9), i]) == 127) and np.abs(aq.astype(int)).max() == 127
    # odd in a, and a power-of-two factor scales s_a only
    aq2, sa2 = oracle.quantize_act(-A)
    assert np.array_equal(aq2, -aq) and np.array_equal(sa2, sa)
    aq3, sa3 = oracle.quantize_act(A * 8.0)
    assert np.array_equal(aq3, aq) and np.array_equal(sa3, sa * 8)
    # a zero row: codes 0, scale 1
    aq4, sa4 = oracle.quantize_act(np.zeros((2, 64)))
    assert np.all(aq4 == 0) and np.all(sa4 == 1.0)


def test_reference_a8_integer_closed_form():
    K, N, M, group = 256, 24, 3, 128
    rng = np.random.default_rng(33)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = np.full((K // group, N), 8, np.uint8)
    s = np.full((K // group, N), 0x3C00, np.uint16)          # 1.0
    aq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    y, mag = oracle.reference_a8(aq, np.ones(M, np.float32), q, s, z, group)
    exact = aq.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(y, exact.astype(np.float64))
    assert np.array_equal(mag, (np.abs(aq.astype(np.int64)) @ np.abs(q.astype(np.int64) - 8)).astype(np.float64))


def test_reference_a8_against_the_16_bit_reference():
    """s_a times the fp16 reference of the codes (exact in fp16) differs from
    the W4A8 reference only by the fp16 rounding of each dequantized weight."""
    K, N, M, group = 512, 40, 4, 128
    q, s, z = oracle.quantize(synthetic.small_weights(K, N, seed=34), group)
    A = synthetic.small_activations(M, K, seed=34).astype(np.float64)
    aq, sa = oracle.quantize_act(A)
    y8, m8 = oracle.reference_a8(aq, sa, q, s, z, group)
    y16, m16 = oracle.reference(aq.astype(np.float16), q, s, z, group)
    sa64 = sa[:, None].astype(np.float64)
    assert np.all(np.abs(y8 - sa64 * y16) <= 2.0 ** -11 * m8 + 1e-12)
    assert np.allclose(m8, sa64 * m16, rtol=2.0 ** -10)
    # and the quantized product is close to the unquantized one
    y, mag = oracle.reference(A.astype(np.float16), q, s, z, group)
    assert np.all(np.abs(y8 - y) <= 0.02 * mag + 1e-3)


def test_worked_example_bf16_and_w4a8():
    """tests/golden/a8_bf16_worked.txt: RNE_bf16 dequantization and the W4A8
    codes and product of the golden group, derived by hand in the file."""
    g = {k: [float(v) for v in vals] for k, vals in _read_golden("a8_bf16_worked.txt").items()}
    q = np.array([0, 4, 6, 10, 15, 9, 5, 8], np.uint8).reshape(8, 1)
    z = np.array([[6]], np.uint8)
    s = np.array([[0x2A66]], np.uint16)
    deq = oracle.from_bf16(oracle.dequantize_bf16(q, s, z, 8)).ravel()
    assert np.array_equal(deq, np.array(g["deq_bf16"]))
    A = np.array([g["a"]])
    aq, sa = oracle.quantize_act(A)
    assert np.array_equal(aq.ravel(), np.array(g["a_q"], dtype=np.int64))
    assert float(sa[0]) == g["s_a"][0]
    y, mag = oracle.reference_a8(aq, sa, q, s, z, 8)
    assert float(y[0, 0]) == g["y"][0] and float(mag[0, 0]) == g["mag"][0]
