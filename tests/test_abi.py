"""Host-side checks of the C ABI (no kernel runs here, no GPU needed).

The library must load, export every entry point declared in
include/w4a16.h, and reject bad arguments on the host with the documented
codes before touching the device.
"""
import ctypes
import os
import re

import pytest

import bit_weight_only_g128_gb300 as w4
from bit_weight_only_g128_gb300 import build as wbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    wbuild.build()
    return w4.lib()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("w4a16_pack", "w4a16_gemm", "w4a16_quantize", "w4a16_unpack",
                 "w4a16_workspace_size", "w4a16_last_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_binding_signatures_cover_the_header():
    assert sorted(w4.SIGNATURES) == declared_symbols()


def test_header_compiles_as_c_and_cpp(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "w4a16.h"\nint main(void){return W4A16_OK;}\n')
    import subprocess
    for comp, ext in (("gcc", "c"), ("g++", "cpp")):
        f = tmp_path / f"t.{ext}"
        f.write_text(src.read_text())
        subprocess.run([comp, "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-c", str(f), "-o", str(tmp_path / f"t_{ext}.o")], check=True)


def test_packed_sizes(lib):
    assert w4.packed_sizes(4096, 4096, 128) == (4096 * 4096 // 2, 2 * 32 * 4096, 32 * 4096 // 2)
    assert w4.packed_sizes(8192, 64, 8192) == (8192 * 64 // 2, 2 * 64, 32)


@pytest.mark.parametrize("K,N,group,code", [
    (4096, 4096, 0, -1), (0, 16, 64, -1), (64, 0, 64, -1),
    (4096, 4100, 128, -2), (4000, 4096, 128, -2), (4096, 4096, 96, -2),
    (4096, 4096, 32, -2), (4096 + 64, 4096, 128, -2), (1 << 21, 16, 64, -2),
])
def test_shape_rules(lib, K, N, group, code):
    w, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    rc = lib.w4a16_packed_sizes(K, N, group, ctypes.byref(w), ctypes.byref(s), ctypes.byref(z))
    assert rc == code
    assert lib.w4a16_last_error()


def _gemm(lib, A=16, W=16, S=16, Z=16, Y=16, M=1, N=64, K=128, group=128, path=0, parts=0,
          ws=256, ws_bytes=1 << 20):
    # fake (never dereferenced) addresses: every failure below is decided on the host
    return lib.w4a16_gemm_ex(A and 0x10000 + A % 16, W and 0x20000 + W % 16,
                             S and 0x30000 + S % 16, Z and 0x40000 + Z % 16, M, N, K, group,
                             Y and 0x50000 + Y % 16, ws and 0x100000 + ws % 256, ws_bytes,
                             path, parts, None)


def test_gemm_argument_errors(lib):
    assert _gemm(lib, A=0) == -1
    assert _gemm(lib, Y=0) == -1
    assert _gemm(lib, M=-1) == -1
    assert _gemm(lib, N=40) == -2
    assert _gemm(lib, K=100) == -2
    assert _gemm(lib, group=48) == -2
    assert _gemm(lib, A=2) == -3
    assert _gemm(lib, Y=8) == -3
    assert _gemm(lib, Z=4) == -3
    assert _gemm(lib, path=7) == -1
    assert _gemm(lib, path=6) == -1
    assert _gemm(lib, path=0x1000 | 1) == -1          # unknown flag bit
    # W4A8 keeps the activations' codes in the workspace: none given
    assert _gemm(lib, path=0x800 | 3, ws=0) == -4
    assert _gemm(lib, path=0x800 | 2, ws=0) == -4
    # bf16 activations: the same host checks (the stream-K variant still
    # needs its workspace)
    assert _gemm(lib, path=0x400 | 4, ws=0) == -4
    assert _gemm(lib, path=0x400 | 1, N=40) == -2
    assert _gemm(lib, path=0x400 | 3, M=16, K=16384, ws=0) == -2
    # fused gate/up epilogue: N must be two halves of whole strips, and a
    # path that does not fuse it keeps the product in the workspace
    assert _gemm(lib, path=0x200 | 1, N=48) == -2
    assert _gemm(lib, path=0x200 | 2, N=80) == -2
    assert _gemm(lib, path=0x200 | 2, ws=0) == -4
    assert _gemm(lib, path=0x200 | 4, ws=0) == -4
    assert _gemm(lib, parts=-1) == -1
    # a K-split tensor launch needs a workspace (K = 512: four 128-k stages)
    assert _gemm(lib, path=2, parts=4, K=512, ws=0) == -4
    assert _gemm(lib, path=1, ws=0) == -4             # decode needs a workspace
    assert _gemm(lib, path=1, ws_bytes=16) == -4
    assert _gemm(lib, path=1, ws=8) == -3             # workspace not 256-byte aligned
    assert _gemm(lib, path=1, K=768, group=192) == -2  # decode: group 64 * 2^j or K
    assert _gemm(lib, path=4, ws=0) == -4             # stream-K needs a workspace
    # the resident variant needs none, and rejects rows that do not fit
    # (16 rows of K = 16384 are 512 KiB of fp16)
    assert _gemm(lib, path=3, M=16, K=16384, ws=0) == -2
    assert _gemm(lib, path=3, M=16, K=16384, group=16384, ws=0) == -2


def test_selftest_rejects_unknown_kinds(lib):
    # decided on the host, before any launch
    assert lib.w4a16_selftest_wait(2, None) == -1
    assert lib.w4a16_selftest_wait(-1, None) == -1


def test_static_weights_flag_matches_the_header():
    text = open(HEADER).read()
    assert re.search(r"#define W4A16_STATIC_WEIGHTS 0x100\b", text)
    assert w4.STATIC_WEIGHTS == 0x100


def test_gemm_m_zero_is_a_noop(lib):
    # M == 0 returns before any pointer is used or any kernel is launched
    assert lib.w4a16_gemm(None, None, None, None, 0, 64, 128, 128, None, None, 0, None) == 0


def test_workspace_sizes(lib):
    # decode path: flags + one fp32 tile (8 or 16 tokens x 128 columns) per
    # CTA; tensor path: counters + one fp32 tile (token tile x 128) per
    # output tile and K range, none without a split
    head = 32768   # flags for up to 8192 CTAs / counters for 2^20 / 128 column blocks
    assert w4.workspace_size(0, 4096, 4096, 128) == 0
    assert w4.workspace_size(64, 4096, 4096, 128, path="tensor", parts=1) == 0
    assert w4.workspace_size(64, 4096, 4096, 128, path="tensor", parts=3) == head + 32 * 3 * 64 * 128 * 4
    assert w4.workspace_size(300, 256, 4096, 128, path="tensor", parts=2) == head + 4 * 2 * 256 * 128 * 4
    assert w4.workspace_size(1, 4096, 4096, 128, path="decode", parts=10) == head + 10 * 8 * 128 * 4
    assert w4.workspace_size(16, 4096, 4096, 128, path="decode", parts=10) == head + 10 * 16 * 128 * 4
    # the decode path's size is the stream-K variant's, whichever variant
    # runs; the resident variant needs none
    for M in (1, 8, 16):
        assert (w4.workspace_size(M, 4096, 4096, 128, path="decode-streamk", parts=10)
                == w4.workspace_size(M, 4096, 4096, 128, path="decode", parts=10))
        assert w4.workspace_size(M, 4096, 4096, 128, path="decode-resident") == 0
    # the CTA count is clamped to the split granules (arguments: M, N, K,
    # group): 32 blocks x 4 groups of 2 atoms
    assert w4.workspace_size(1, 4096, 512, 128, path="decode", parts=1000) == head + 128 * 8 * 128 * 4
    # groups of 8 atoms or more split every 8 atoms: 32 blocks x 1, 4 x 8
    assert w4.workspace_size(1, 4096, 512, 512, path="decode", parts=1000) == head + 32 * 8 * 128 * 4
    assert w4.workspace_size(1, 512, 4096, 1024, path="decode", parts=1000) == head + 32 * 8 * 128 * 4
    # one group per column (K not a power-of-two number of atoms): any 64-k
    # boundary, 4 blocks x 5 atoms
    assert w4.workspace_size(1, 512, 320, 320, path="decode", parts=1000) == head + 20 * 8 * 128 * 4
    # and never above 8192 CTAs
    assert w4.workspace_size(1, 65536, 4096, 64, path="decode", parts=20000) == head + 8192 * 8 * 128 * 4


def test_silu_mul_workspace_sizes(lib):
    # the product [rows][N] fp16 after the path's own scratch, at a 256-byte
    # boundary, and never inside the 32 KiB flag/counter area (which a later
    # call may use); none for the resident variant, which fuses the epilogue
    head = 32768
    assert w4.workspace_size(64, 4096, 4096, 128, path="tensor", parts=1,
                             silu_mul=True) == head + 64 * 4096 * 2
    base = head + 32 * 3 * 64 * 128 * 4
    assert w4.workspace_size(64, 4096, 4096, 128, path="tensor", parts=3,
                             silu_mul=True) == (base + 255) // 256 * 256 + 64 * 4096 * 2
    assert w4.workspace_size(300, 352, 4096, 128, path="tensor", parts=1,
                             silu_mul=True) == head + 300 * 352 * 2
    assert w4.workspace_size(16, 4096, 4096, 128, path="decode-resident", silu_mul=True) == 0
    for M, rows in ((1, 1), (16, 16), (40, 16)):
        base = w4.workspace_size(M, 4096, 4096, 128, path="decode-streamk", parts=10)
        for path in ("decode", "decode-streamk"):
            assert w4.workspace_size(M, 4096, 4096, 128, path=path, parts=10,
                                     silu_mul=True) == (base + 255) // 256 * 256 + rows * 4096 * 2
    assert w4.SILU_MUL == 0x200 and w4.BF16 == 0x400
    assert re.search(r"#define W4A16_BF16 0x400\b", open(HEADER).read())
    # bf16 activations change no size
    for path, parts in (("tensor", 3), ("decode", 10), ("decode-streamk", 10)):
        b = ctypes.c_size_t()
        for flags in (0, 0x200):
            assert lib.w4a16_workspace_size_ex(16, 4096, 4096, 128, w4._PATHS[path] | flags, parts,
                                               ctypes.byref(b)) == 0
            plain = b.value
            assert lib.w4a16_workspace_size_ex(16, 4096, 4096, 128, w4._PATHS[path] | flags | 0x400,
                                               parts, ctypes.byref(b)) == 0
            assert b.value == plain
    assert re.search(r"#define W4A16_SILU_MUL 0x200\b", open(HEADER).read())


def test_w4a8_workspace_and_quantize_act_errors(lib):
    head = 32768
    # codes [M][K] 16-bit then scales [M], after the path's scratch (and at
    # least after the flag area), at 256-byte boundaries
    def up(b):
        return (b + 255) // 256 * 256
    M, N, K = 16, 4096, 4096
    assert w4.workspace_size(M, N, K, 128, path="decode-resident", a8=True) == up(head + M * K * 2) + M * 4
    base = w4.workspace_size(M, N, K, 128, path="tensor", parts=3)
    assert w4.workspace_size(M, N, K, 128, path="tensor", parts=3, a8=True) == up(up(base) + M * K * 2) + M * 4
    both = w4.workspace_size(M, N, K, 128, path="decode-streamk", parts=10, silu_mul=True)
    assert w4.workspace_size(M, N, K, 128, path="decode-streamk", parts=10, silu_mul=True,
                             a8=True) == up(up(both) + M * K * 2) + M * 4
    assert w4.workspace_size(40, N, K, 128, path="decode", parts=10, a8=True) == \
        up(up(w4.workspace_size(40, N, K, 128, path="decode", parts=10)) + 40 * K * 2) + 40 * 4
    A, Q, S = 0x10000, 0x20000, 0x30000
    assert lib.w4a16_quantize_act(A, -1, 64, 0, Q, S, None) == -1
    assert lib.w4a16_quantize_act(A, 4, 60, 0, Q, S, None) == -2
    assert lib.w4a16_quantize_act(A, 4, 65536 + 64, 0, Q, S, None) == -2
    assert _gemm(lib, path=0x800 | 2, K=65536 + 64, group=64) == -2
    assert lib.w4a16_quantize_act(A, 4, 64, 0x200, Q, S, None) == -1
    assert lib.w4a16_quantize_act(A + 8, 4, 64, 0, Q, S, None) == -3
    assert lib.w4a16_quantize_act(A, 4, 64, 0, Q + 4, S, None) == -3
    assert lib.w4a16_quantize_act(None, 4, 64, 0, Q, S, None) == -1
    assert lib.w4a16_quantize_act(None, 0, 64, 0, None, None, None) == 0
    assert w4.ACT_A8 == 0x800 and re.search(r"#define W4A16_ACT_A8 0x800\b", open(HEADER).read())


def test_path_constants_match_the_header():
    text = open(HEADER).read()
    for name, value in (("W4A16_PATH_AUTO", 0), ("W4A16_PATH_DECODE", 1), ("W4A16_PATH_TENSOR", 2),
                        ("W4A16_PATH_DECODE_RESIDENT", 3), ("W4A16_PATH_DECODE_STREAMK", 4)):
        assert re.search(rf"#define {name} {value}\b", text), name
    assert (w4.PATH_AUTO, w4.PATH_DECODE, w4.PATH_TENSOR, w4.PATH_DECODE_RESIDENT,
            w4.PATH_DECODE_STREAMK) == (0, 1, 2, 3, 4)


def test_plan_follows_the_measured_path_rules(lib):
    """w4a16_plan (host only) reports the paths of the measured dispatch
    rules: decode up to 16 rows, on wide layers (N >= 16384) of at most 2^28
    weights up to 24 rows; the CTA-pair kernel on such wide layers at 65-128
    rows, on every wide layer at 193-255 rows, and from 256
    rows where the pairs make at least 80 CTAs; single-SM tensor-core tiles
    otherwise; tensor cores whenever the decode kernel does not take the
    group size."""
    def path(M, N, K, g=128):
        return w4.plan(M, N, K, g)[0]
    assert path(1, 12288, 4096).startswith("decode")
    assert path(16, 4096, 4096).startswith("decode")
    assert path(24, 22016, 4096).startswith("decode")        # 7B gate_up: two decode passes
    assert path(24, 27648, 5120).startswith("decode")        # 13B gate_up
    assert path(25, 27648, 5120) == "tensor"
    assert path(32, 22016, 4096) == "tensor"
    assert path(16, 57344, 8192).startswith("decode")        # 70B gate_up
    assert path(17, 57344, 8192) == "tensor"                 # above 2^28 weights
    assert path(20, 15360, 5120) == "tensor"                 # 13B qkv
    assert path(128, 57344, 8192) == "tensor"                # above 2^28 weights: one SM
    assert path(128, 22016, 4096) == "tensor-pair"           # 7B gate_up, 65-128 rows
    assert path(65, 27648, 5120) == "tensor-pair"            # 13B gate_up
    assert path(64, 27648, 5120) == "tensor"
    assert path(128, 15360, 5120) == "tensor"                # narrower than 16384
    assert path(129, 22016, 4096) == "tensor"
    assert path(192, 22016, 4096) == "tensor"
    assert path(193, 22016, 4096) == "tensor-pair"           # wide layers, 193-255 rows
    assert path(255, 57344, 8192) == "tensor-pair"
    assert path(224, 15360, 5120) == "tensor"                # narrower than 16384
    assert path(256, 10240, 8192) == "tensor-pair"           # 2 x 40 pair CTAs
    assert path(256, 8192, 8192) == "tensor"                 # 2 x 32: too few
    assert path(512, 4096, 11008) == "tensor"                # 2 x 16 x 2
    assert path(512, 5120, 5120) == "tensor-pair"            # 2 x 20 x 2
    assert path(512, 57344, 8192) == "tensor-pair"
    assert path(4096, 8192, 8192) == "tensor-pair"
    assert path(4096, 4096, 4096) == "tensor-pair"
    assert path(8, 256, 768, 192) == "tensor"                # group 192: decode does not take it
    assert path(8, 256, 768, 768).startswith("decode")       # group == K does
