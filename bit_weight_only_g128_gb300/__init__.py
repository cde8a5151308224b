"""GB300 (sm_103a) W4A16 group-quantized linear layer: Python binding.

A thin ctypes layer over the C ABI in include/w4a16.h (libw4a16.so, built
in-tree by ``build.build()``). PyTorch supplies device memory and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels. There is no fallback: if the library is missing or a call
fails, an exception is raised.

The operation (compressed-tensors PR #269 "Some fixes for AWQ", reply
defining w4a16): Y[M,N] fp16 = A[M,K] fp16 . dequant(W)[K,N], with W
quantized asymmetrically per group of `group` input channels (the AWQ-g128
format of vLLM PR #1032 "Implement AWQ quantization support for LLaMA").
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional, Tuple

import torch

from .build import LIB as _BUILT_LIB

# the library to load: W4A16_LIBRARY (for example the bounds-checked build),
# else the in-tree build
LIB_PATH = os.environ.get("W4A16_LIBRARY") or _BUILT_LIB

PATH_AUTO, PATH_DECODE, PATH_TENSOR = 0, 1, 2
PATH_DECODE_RESIDENT, PATH_DECODE_STREAMK, PATH_TENSOR_PAIR = 3, 4, 5
_PATHS = {"auto": PATH_AUTO, "decode": PATH_DECODE, "tensor": PATH_TENSOR,
          "decode-resident": PATH_DECODE_RESIDENT, "decode-streamk": PATH_DECODE_STREAMK,
          "tensor-pair": PATH_TENSOR_PAIR}
STATIC_WEIGHTS = 0x100  # W4A16_STATIC_WEIGHTS
SILU_MUL = 0x200        # W4A16_SILU_MUL
BF16 = 0x400            # W4A16_BF16
ACT_A8 = 0x800          # W4A16_ACT_A8

ERRORS = {
    -1: "INVALID_ARG", -2: "UNSUPPORTED_SHAPE", -3: "MISALIGNED",
    -4: "WORKSPACE_TOO_SMALL", -5: "CUDA_ERROR", -6: "DEVICE_CHECK",
}

# every symbol declared in include/w4a16.h, with its ctypes signature
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_PSZ = ctypes.POINTER(ctypes.c_size_t)
_PI = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "w4a16_last_error": (ctypes.c_char_p, []),
    "w4a16_version": (_I, []),
    "w4a16_packed_sizes": (_I, [_I, _I, _I, _PSZ, _PSZ, _PSZ]),
    "w4a16_quantize": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "w4a16_pack": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "w4a16_unpack": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "w4a16_dequantize": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "w4a16_dequantize_bf16": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "w4a16_quantize_act": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "w4a16_workspace_size": (_I, [_I, _I, _I, _I, _PSZ]),
    "w4a16_workspace_size_ex": (_I, [_I, _I, _I, _I, _I, _I, _PSZ]),
    "w4a16_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "w4a16_gemm_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _SZ, _I, _I, _P]),
    "w4a16_plan": (_I, [_I, _I, _I, _I, _PI, _PI]),
    "w4a16_tc_config": (_I, [_I, _I, _I, _PI, _I]),
    "w4a16_gemm_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "w4a16_device_status": (_I, [_P]),
    "w4a16_selftest_wait": (_I, [_I, _P]),
}

_lock = threading.Lock()
_lib = None


class W4A16Error(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {message}")


def lib() -> ctypes.CDLL:
    """Load libw4a16.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m bit_weight_only_g128_gb300.build` (needs nvcc)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != 0:
        msg = lib().w4a16_last_error().decode(errors="replace")
        raise W4A16Error(rc, where, msg)


def _stream(stream: Optional[torch.cuda.Stream], device: Optional[int] = None) -> int:
    """The cudaStream_t of `stream`, or of the current stream of `device`
    (default: the current device)."""
    if stream is not None:
        return stream.cuda_stream
    if device is None:
        device = torch.cuda.current_device()
    return torch._C._cuda_getCurrentRawStream(device)


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


@dataclasses.dataclass
class PackedWeight:
    """Packed int4 weight of one linear layer, resident on the device."""
    Wq: torch.Tensor       # int32 [K*N/8]
    Sp: torch.Tensor       # float16 [K/group * N]
    Zp: torch.Tensor       # int32 [K/group * N / 8]
    K: int
    N: int
    group: int

    @property
    def nbytes(self) -> int:
        return self.Wq.numel() * 4 + self.Sp.numel() * 2 + self.Zp.numel() * 4


def packed_sizes(K: int, N: int, group: int) -> Tuple[int, int, int]:
    w, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().w4a16_packed_sizes(K, N, group, ctypes.byref(w), ctypes.byref(s),
                                    ctypes.byref(z)), "w4a16_packed_sizes")
    return w.value, s.value, z.value


def quantize(W: torch.Tensor, group: int, stream=None):
    """fp32 W [K, N] (device) -> (q uint8 [K,N], s fp16 [G,N], z uint8 [G,N])."""
    K, N = W.shape
    G = K // group if group > 0 else 0
    q = torch.empty((K, N), dtype=torch.uint8, device=W.device)
    s = torch.empty((G, N), dtype=torch.float16, device=W.device)
    z = torch.empty((G, N), dtype=torch.uint8, device=W.device)
    _check(lib().w4a16_quantize(_dev(W, torch.float32, "W"), K, N, group, q.data_ptr(),
                                s.data_ptr(), z.data_ptr(), _stream(stream)), "w4a16_quantize")
    return q, s, z


def pack(q: torch.Tensor, s: torch.Tensor, z: torch.Tensor, group: int, stream=None) -> PackedWeight:
    """Interchange (q, s, z) -> PackedWeight in the library's device layout."""
    K, N = q.shape
    wb, sb, zb = packed_sizes(K, N, group)
    dev = q.device
    Wq = torch.empty(wb // 4, dtype=torch.int32, device=dev)
    Sp = torch.empty(sb // 2, dtype=torch.float16, device=dev)
    Zp = torch.empty(zb // 4, dtype=torch.int32, device=dev)
    _check(lib().w4a16_pack(_dev(q, torch.uint8, "q"), _dev(s, torch.float16, "s"),
                            _dev(z, torch.uint8, "z"), K, N, group, Wq.data_ptr(),
                            Sp.data_ptr(), Zp.data_ptr(), _stream(stream)), "w4a16_pack")
    return PackedWeight(Wq, Sp, Zp, K, N, group)


def quantize_pack(W: torch.Tensor, group: int, stream=None) -> PackedWeight:
    q, s, z = quantize(W, group, stream)
    return pack(q, s, z, group, stream)


def unpack(pw: PackedWeight, stream=None):
    dev = pw.Wq.device
    G = pw.K // pw.group
    q = torch.empty((pw.K, pw.N), dtype=torch.uint8, device=dev)
    s = torch.empty((G, pw.N), dtype=torch.float16, device=dev)
    z = torch.empty((G, pw.N), dtype=torch.uint8, device=dev)
    _check(lib().w4a16_unpack(pw.Wq.data_ptr(), pw.Sp.data_ptr(), pw.Zp.data_ptr(), pw.K, pw.N,
                              pw.group, q.data_ptr(), s.data_ptr(), z.data_ptr(),
                              _stream(stream)), "w4a16_unpack")
    return q, s, z


def dequantize(pw: PackedWeight, stream=None, dtype: torch.dtype = torch.float16) -> torch.Tensor:
    """deq [K, N] = RNE((q - z) * s) in fp16, or in bf16 (the tensor-core
    path's operand for bf16 activations)."""
    if dtype not in (torch.float16, torch.bfloat16):
        raise ValueError(f"dtype must be float16 or bfloat16, got {dtype}")
    deq = torch.empty((pw.K, pw.N), dtype=dtype, device=pw.Wq.device)
    fn = lib().w4a16_dequantize_bf16 if dtype == torch.bfloat16 else lib().w4a16_dequantize
    _check(fn(pw.Wq.data_ptr(), pw.Sp.data_ptr(), pw.Zp.data_ptr(), pw.K, pw.N, pw.group,
              deq.data_ptr(), _stream(stream)), "w4a16_dequantize")
    return deq


_ws_sizes = {}


def workspace_size(M: int, N: int, K: int, group: int, path: str = "auto", parts: int = 0,
                   silu_mul: bool = False, a8: bool = False, device: Optional[int] = None) -> int:
    """Scratch bytes a gemm call with these arguments needs on the current
    device (cached per device and arguments: the size depends on nothing else)."""
    dev = device if device is not None else (
        torch.cuda.current_device() if torch.cuda.is_available() else -1)
    key = (dev, M, N, K, group, path, parts, silu_mul, a8)
    size = _ws_sizes.get(key)
    if size is None:
        b = ctypes.c_size_t()
        flags = (SILU_MUL if silu_mul else 0) | (ACT_A8 if a8 else 0)
        _check(lib().w4a16_workspace_size_ex(M, N, K, group, _PATHS[path] | flags, parts,
                                             ctypes.byref(b)), "w4a16_workspace_size")
        size = _ws_sizes[key] = b.value
    return size


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace (every call leaves it zeroed)."""
    return torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=device or "cuda")


# workspaces of gemm calls that pass none: one per (device, stream), grown on
# demand. Calls on one stream run one after another, so they can share one;
# calls on different streams get different ones.
_stream_ws = {}


def stream_workspace(nbytes: int, device: int, stream: int) -> torch.Tensor:
    """The cached workspace of the stream `stream` (a cudaStream_t) on device
    index `device`, at least `nbytes` long (a larger zero-filled one replaces
    it when it is too small)."""
    key = (device, stream)
    ws = _stream_ws.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = _stream_ws[key] = new_workspace(nbytes, torch.device("cuda", device))
    return ws


def plan(M: int, N: int, K: int, group: int) -> Tuple[str, int]:
    """(path, decode CTA count) the library picks for this problem."""
    p, c = ctypes.c_int(), ctypes.c_int()
    _check(lib().w4a16_plan(M, N, K, group, ctypes.byref(p), ctypes.byref(c)), "w4a16_plan")
    return {v: k for k, v in _PATHS.items()}[p.value], c.value


TC_CONFIG_KEYS = ("token_tile", "stage_atoms", "act_slots", "code_slots", "dq_slots",
                  "dequant_groups", "smem_bytes", "ctas_per_sm")


def tc_config(M: int, K: int, group: int, pair: bool = False) -> dict:
    """The one-SM tensor-core kernel's configuration for M rows, or with
    `pair` the CTA-pair kernel's (per CTA; ctas_per_sm 1) (host-only)."""
    out = (ctypes.c_int * 15)()
    _check(lib().w4a16_tc_config(M, K, group, out, 15), "w4a16_tc_config")
    vals = list(out)
    return dict(zip(TC_CONFIG_KEYS, vals[8:15] + [1] if pair else vals[:8]))


def gemm(A: torch.Tensor, pw: PackedWeight, out: Optional[torch.Tensor] = None,
         path: str = "auto", parts: int = 0, workspace: Optional[torch.Tensor] = None,
         stream=None, static_weights: bool = False, silu_mul: bool = False,
         a8: bool = False) -> torch.Tensor:
    """Y [M, N] = A [M, K] . dequant(pw), on the current stream; A and Y are
    both fp16 or both bf16 (W4A16_BF16, chosen by A's dtype).

    `workspace` must be zero-filled before its first use (new_workspace);
    without one, the call uses the cached workspace of its stream
    (stream_workspace), allocated on the first call that needs it and grown
    when a call needs more.
    `static_weights` (W4A16_STATIC_WEIGHTS): the kernel may read pw while the
    work queued before it on the stream drains; pw must not be written by
    that work. `silu_mul` (W4A16_SILU_MUL): pw's columns are [gate | up] and
    Y [M, N/2] = silu(gate) * up. `a8` (W4A16_ACT_A8): W4A8, the activations
    are quantized per row to int8 inside the call.
    """
    M, K = A.shape
    if K != pw.K:
        raise ValueError(f"A has K={K}, weight has K={pw.K}")
    dt = A.dtype if A.dtype in (torch.float16, torch.bfloat16) else torch.float16
    a_ptr = _dev(A, dt, "A")
    dev = A.device.index
    if out is None:
        out = torch.empty((M, pw.N // 2 if silu_mul else pw.N), dtype=dt, device=A.device)
    y_ptr = _dev(out, dt, "out")
    st = _stream(stream, dev)
    ws_ptr, ws_bytes = None, 0
    need = workspace_size(M, pw.N, pw.K, pw.group, path, parts, silu_mul, a8, dev)
    if need:
        if workspace is None:
            workspace = stream_workspace(need, dev, st)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = lib().w4a16_gemm_ex(a_ptr, pw.Wq.data_ptr(), pw.Sp.data_ptr(), pw.Zp.data_ptr(), M,
                             pw.N, pw.K, pw.group, y_ptr, ws_ptr, ws_bytes,
                             _PATHS[path] | (STATIC_WEIGHTS if static_weights else 0)
                             | (SILU_MUL if silu_mul else 0) | (ACT_A8 if a8 else 0)
                             | (BF16 if dt == torch.bfloat16 else 0), parts, st)
    if rc:
        _check(rc, "w4a16_gemm")
    return out


def quantize_act(A: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """W4A8 activation quantization: A [M, K] fp16/bf16 -> (a_q int8 [M, K],
    s_a float32 [M]), the rule W4A16_ACT_A8 applies inside gemm."""
    M, K = A.shape
    dt = A.dtype if A.dtype in (torch.float16, torch.bfloat16) else torch.float16
    aq = torch.empty((M, K), dtype=torch.int8, device=A.device)
    sa = torch.empty((M,), dtype=torch.float32, device=A.device)
    _check(lib().w4a16_quantize_act(_dev(A, dt, "A"), M, K, BF16 if dt == torch.bfloat16 else 0,
                                    aq.data_ptr(), sa.data_ptr(), _stream(stream)),
           "w4a16_quantize_act")
    return aq, sa


def gemm_noalloc(A: torch.Tensor, pw: PackedWeight, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Decode-path Y = A . dequant(pw) through w4a16_gemm_noalloc: no workspace;
    the library's own device scratch array is used instead (see the header)."""
    M, K = A.shape
    if K != pw.K:
        raise ValueError(f"A has K={K}, weight has K={pw.K}")
    if out is None:
        out = torch.empty((M, pw.N), dtype=torch.float16, device=A.device)
    _check(lib().w4a16_gemm_noalloc(_dev(A, torch.float16, "A"), pw.Wq.data_ptr(),
                                    pw.Sp.data_ptr(), pw.Zp.data_ptr(), M, pw.N, pw.K, pw.group,
                                    _dev(out, torch.float16, "out"), _stream(stream)),
           "w4a16_gemm_noalloc")
    return out


def selftest_wait(which: int, stream=None) -> None:
    """Launch the bounded-wait self-test (0: flag wait, 1: mbarrier wait); the
    next device_status() raises W4A16Error with DEVICE_CHECK."""
    _check(lib().w4a16_selftest_wait(which, _stream(stream)), "w4a16_selftest_wait")


def device_status(stream=None) -> None:
    """Synchronize and raise if a kernel reported an error on the device."""
    _check(lib().w4a16_device_status(_stream(stream)), "w4a16_device_status")
