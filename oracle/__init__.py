"""CPU oracle for the W4A16 group-quantized linear layer (ctypes driver).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by
the bench's CPU-baseline leg, never by the CUDA library or its binding. The
arithmetic lives in ``w4a16_oracle.c`` (plain C, fp64 where it accumulates);
this module only builds it with gcc, marshals numpy arrays and calls it.

Sources: compressed-tensors PR #269 "Some fixes for AWQ" (the asymmetric
pseudo_quantize_tensor rule it aligns with; the reply defining w4a16 as fp16
inputs times int4-quantized weights giving fp16 outputs). The rule's formulas
are s = (max-min)/15, z = round(-min/s), q = clamp(round(w/s)+z, 0, 15) and
dequant = (q-z)*s; the tolerance of a product is 2^-9*sum|a*w| + 1e-3.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if force or not fresh:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = {
    "oracle_half_to_double": (ctypes.c_double, [ctypes.c_uint16]),
    "oracle_double_to_half": (ctypes.c_uint16, [ctypes.c_double]),
    "oracle_doubles_to_half": (None, [_P, _SZ, _P]),
    "oracle_halves_to_double": (None, [_P, _SZ, _P]),
    "oracle_quantize": (None, [_P, _I, _I, _I, _P, _P, _P]),
    "oracle_dequantize": (None, [_P, _P, _P, _I, _I, _I, _P]),
    "oracle_matmul": (None, [_P, _P, _I, _I, _I, _P, _P]),
    "oracle_check": (ctypes.c_double, [_P, _P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "oracle_pack": (None, [_P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "oracle_unpack": (None, [_P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "oracle_threads": (_I, []),
    "oracle_silu": (ctypes.c_double, [ctypes.c_double]),
    "oracle_silu_mul": (None, [_P, _P, _I, _I, _P, _P]),
    "oracle_check_bound": (ctypes.c_double, [_P, _P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "oracle_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
    "oracle_double_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
    "oracle_doubles_to_bf16": (None, [_P, _SZ, _P]),
    "oracle_bf16s_to_double": (None, [_P, _SZ, _P]),
    "oracle_dequantize_bf16": (None, [_P, _P, _P, _I, _I, _I, _P]),
    "oracle_matmul_bf16": (None, [_P, _P, _I, _I, _I, _P, _P]),
    "oracle_check_bf16": (ctypes.c_double, [_P, _P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "oracle_silu_mul_bf16": (None, [_P, _P, _I, _I, _P, _P]),
    "oracle_check_bound_bf16": (ctypes.c_double, [_P, _P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "oracle_quantize_act": (None, [_P, _I, _I, _P, _P]),
    "oracle_reference_a8": (None, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            handle = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_half_bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def threads() -> int:
    return int(lib().oracle_threads())


def to_half(x) -> np.ndarray:
    """Round doubles to binary16 (ties to even); returns uint16 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    shape = x.shape
    x = np.ascontiguousarray(x.reshape(-1))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_doubles_to_half(_ptr(x), x.size, _ptr(out))
    return out.reshape(shape)


def from_half(h) -> np.ndarray:
    """Exact value of binary16 bit patterns as doubles."""
    h = np.asarray(h)
    shape = h.shape
    h = _as_half_bits(h.reshape(-1))
    out = np.empty(h.shape, dtype=np.float64)
    lib().oracle_halves_to_double(_ptr(h), h.size, _ptr(out))
    return out.reshape(shape)


def quantize(W: np.ndarray, group: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """W float32 [K, N] -> (q u8 [K,N], s fp16 bits u16 [G,N], z u8 [G,N])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    K, N = W.shape
    assert group > 0 and K % group == 0
    G = K // group
    q = np.empty((K, N), np.uint8)
    s = np.empty((G, N), np.uint16)
    z = np.empty((G, N), np.uint8)
    lib().oracle_quantize(_ptr(W), K, N, group, _ptr(q), _ptr(s), _ptr(z))
    return q, s, z


def dequantize(q: np.ndarray, s: np.ndarray, z: np.ndarray, group: int) -> np.ndarray:
    """(q, s, z) -> deq fp16 bits u16 [K, N] = RNE_fp16((q - z) * s)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _as_half_bits(s)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    K, N = q.shape
    assert s.shape == (K // group, N) and z.shape == s.shape
    deq = np.empty((K, N), np.uint16)
    lib().oracle_dequantize(_ptr(q), _ptr(s), _ptr(z), K, N, group, _ptr(deq))
    return deq


def matmul(A, B) -> Tuple[np.ndarray, np.ndarray]:
    """fp16 A [M,K] times fp16 B [K,N] in fp64 -> (y [M,N], sum|a*b| [M,N])."""
    A = _as_half_bits(A)
    B = _as_half_bits(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    y = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    lib().oracle_matmul(_ptr(A), _ptr(B), M, N, K, _ptr(y), _ptr(mag))
    return y, mag


def reference(A, q, s, z, group) -> Tuple[np.ndarray, np.ndarray]:
    """The W4A16 linear layer: y = A . dequant(q, s, z), in fp64."""
    return matmul(A, dequantize(q, s, z, group))


def check(Y, y_ref: np.ndarray, mag: np.ndarray) -> Tuple[float, int]:
    """max |Y - y_ref| / (2^-9 * mag + 1e-3) over all elements, and its index."""
    Y = _as_half_bits(Y)
    y_ref = np.ascontiguousarray(y_ref, dtype=np.float64)
    mag = np.ascontiguousarray(mag, dtype=np.float64)
    assert Y.shape == y_ref.shape == mag.shape
    wi = _SZ(0)
    r = lib().oracle_check(_ptr(Y), _ptr(y_ref), _ptr(mag), Y.size, ctypes.byref(wi))
    return float(r), int(wi.value)


def packed_shapes(K: int, N: int, group: int):
    G = K // group
    return (K * N // 8,), (G * N,), (G * N // 8,)


def pack(q: np.ndarray, z: np.ndarray, s: np.ndarray, group: int):
    """(q, z, s) -> (Wp u32, Sp u16, Zp u32) in the packed device layout."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    s = _as_half_bits(s)
    K, N = q.shape
    assert N % 16 == 0 and K % 64 == 0 and K % group == 0
    sw, ss, sz = packed_shapes(K, N, group)
    Wp = np.empty(sw, np.uint32)
    Sp = np.empty(ss, np.uint16)
    Zp = np.empty(sz, np.uint32)
    lib().oracle_pack(_ptr(q), _ptr(z), _ptr(s), K, N, group, _ptr(Wp), _ptr(Sp), _ptr(Zp))
    return Wp, Sp, Zp


def unpack(Wp, Sp, Zp, K: int, N: int, group: int):
    """Inverse of pack: -> (q u8 [K,N], s u16 [G,N], z u8 [G,N])."""
    Wp = np.ascontiguousarray(Wp, dtype=np.uint32)
    Sp = _as_half_bits(Sp)
    Zp = np.ascontiguousarray(Zp, dtype=np.uint32)
    G = K // group
    q = np.empty((K, N), np.uint8)
    s = np.empty((G, N), np.uint16)
    z = np.empty((G, N), np.uint8)
    lib().oracle_unpack(_ptr(Wp), _ptr(Sp), _ptr(Zp), K, N, group, _ptr(q), _ptr(s), _ptr(z))
    return q, s, z


def silu(x: float) -> float:
    """silu(x) = x / (1 + exp(-x)) in fp64."""
    return float(lib().oracle_silu(float(x)))


def silu_mul(y: np.ndarray, mag: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Fused gate/up epilogue of a product y [M, N] = [gate | up]:
    (out [M, N/2] = silu(gate) * up, bound [M, N/2]) in fp64 (lmdeploy issue
    #2274, "Modification": gate and up fused into one weight, SiLU fused)."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    mag = np.ascontiguousarray(mag, dtype=np.float64)
    M, N = y.shape
    assert N % 2 == 0 and mag.shape == y.shape
    out = np.empty((M, N // 2), np.float64)
    bound = np.empty((M, N // 2), np.float64)
    lib().oracle_silu_mul(_ptr(y), _ptr(mag), M, N, _ptr(out), _ptr(bound))
    return out, bound


def check_bound(Y, ref: np.ndarray, bound: np.ndarray) -> Tuple[float, int]:
    """max |Y - ref| / bound over all elements, and its index."""
    Y = _as_half_bits(Y)
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    bound = np.ascontiguousarray(bound, dtype=np.float64)
    assert Y.shape == ref.shape == bound.shape
    wi = _SZ(0)
    r = lib().oracle_check_bound(_ptr(Y), _ptr(ref), _ptr(bound), Y.size, ctypes.byref(wi))
    return float(r), int(wi.value)


# ---------------------------------------------------------------- bf16
# compressed-tensors PR #269 "Some fixes for AWQ": W4A16 keeps the
# activations as unquantized 16-bit floats, and a reply names an API taking
# fp32, bf16 or fp16 activations. Readings (see w4a16_oracle.c): A and Y
# bf16 with the same quantized weights; dequant = RNE_bf16((q - z) * s16);
# tolerance 2^-6 * sum|a*w| + 1e-3 (four units of bf16 rounding).

def _as_u16(a) -> np.ndarray:
    a = np.asarray(a)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def to_bf16(x) -> np.ndarray:
    """Round doubles to bfloat16 (ties to even); returns uint16 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    shape = x.shape
    x = np.ascontiguousarray(x.reshape(-1))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_doubles_to_bf16(_ptr(x), x.size, _ptr(out))
    return out.reshape(shape)


def from_bf16(h) -> np.ndarray:
    """Exact value of bfloat16 bit patterns as doubles."""
    h = np.asarray(h)
    shape = h.shape
    h = _as_u16(h.reshape(-1))
    out = np.empty(h.shape, dtype=np.float64)
    lib().oracle_bf16s_to_double(_ptr(h), h.size, _ptr(out))
    return out.reshape(shape)


def dequantize_bf16(q: np.ndarray, s: np.ndarray, z: np.ndarray, group: int) -> np.ndarray:
    """(q, s, z) -> deq bf16 bits u16 [K, N] = RNE_bf16((q - z) * s)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _as_half_bits(s)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    K, N = q.shape
    assert s.shape == (K // group, N) and z.shape == s.shape
    deq = np.empty((K, N), np.uint16)
    lib().oracle_dequantize_bf16(_ptr(q), _ptr(s), _ptr(z), K, N, group, _ptr(deq))
    return deq


def matmul_bf16(A, B) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 A [M,K] times bf16 B [K,N] in fp64 -> (y [M,N], sum|a*b| [M,N])."""
    A = _as_u16(A)
    B = _as_u16(B)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    y = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    lib().oracle_matmul_bf16(_ptr(A), _ptr(B), M, N, K, _ptr(y), _ptr(mag))
    return y, mag


def reference_bf16(A, q, s, z, group) -> Tuple[np.ndarray, np.ndarray]:
    """The layer with bf16 activations: y = A . RNE_bf16(dequant), in fp64."""
    return matmul_bf16(A, dequantize_bf16(q, s, z, group))


def check_bf16(Y, y_ref: np.ndarray, mag: np.ndarray) -> Tuple[float, int]:
    """max |Y - y_ref| / (2^-6 * mag + 1e-3) over bf16 results, and its index."""
    Y = _as_u16(Y)
    y_ref = np.ascontiguousarray(y_ref, dtype=np.float64)
    mag = np.ascontiguousarray(mag, dtype=np.float64)
    assert Y.shape == y_ref.shape == mag.shape
    wi = _SZ(0)
    r = lib().oracle_check_bf16(_ptr(Y), _ptr(y_ref), _ptr(mag), Y.size, ctypes.byref(wi))
    return float(r), int(wi.value)


def silu_mul_bf16(y: np.ndarray, mag: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """silu_mul of a bf16-activation product, with the bound propagated from
    the bf16 tolerance."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    mag = np.ascontiguousarray(mag, dtype=np.float64)
    M, N = y.shape
    assert N % 2 == 0 and mag.shape == y.shape
    out = np.empty((M, N // 2), np.float64)
    bound = np.empty((M, N // 2), np.float64)
    lib().oracle_silu_mul_bf16(_ptr(y), _ptr(mag), M, N, _ptr(out), _ptr(bound))
    return out, bound


def check_bound_bf16(Y, ref: np.ndarray, bound: np.ndarray) -> Tuple[float, int]:
    """max |Y - ref| / bound over bf16 results, and its index."""
    Y = _as_u16(Y)
    ref = np.ascontiguousarray(ref, dtype=np.float64)
    bound = np.ascontiguousarray(bound, dtype=np.float64)
    assert Y.shape == ref.shape == bound.shape
    wi = _SZ(0)
    r = lib().oracle_check_bound_bf16(_ptr(Y), _ptr(ref), _ptr(bound), Y.size, ctypes.byref(wi))
    return float(r), int(wi.value)


# ---------------------------------------------------------------- W4A8
# compressed-tensors PR #269, the Arm example: fp16 in, activations quantized
# to 8 bits inside the operation, 8-bit x 4-bit product, fp16 out (lmdeploy
# issue #2274: W4A8 with online activation quantization). Readings (see
# w4a16_oracle.c): dynamic symmetric per-token int8, s_a = amax/127 in fp32,
# integer group dot products scaled per group and per row.

def quantize_act(A_values: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Activation values [M, K] (exact fp16/bf16 values as doubles) ->
    (a_q int8 [M, K], s_a float32 [M])."""
    A = np.ascontiguousarray(A_values, dtype=np.float64)
    M, K = A.shape
    aq = np.empty((M, K), np.int8)
    sa = np.empty((M,), np.float32)
    lib().oracle_quantize_act(_ptr(A), M, K, _ptr(aq), _ptr(sa))
    return aq, sa


def reference_a8(aq, sa, q, s, z, group) -> Tuple[np.ndarray, np.ndarray]:
    """y = s_a * sum_g s * sum_k a_q (q - z) and its magnitude sum, in fp64."""
    aq = np.ascontiguousarray(aq, dtype=np.int8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _as_half_bits(s)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    M, K = aq.shape
    N = q.shape[1]
    assert q.shape == (K, N) and s.shape == (K // group, N) and z.shape == s.shape and sa.shape == (M,)
    y = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    lib().oracle_reference_a8(_ptr(aq), _ptr(sa), _ptr(q), _ptr(s), _ptr(z), M, N, K, group,
                              _ptr(y), _ptr(mag))
    return y, mag
