"""The Python binding's own checks (no GPU): it rejects host tensors, wrong
dtypes and mismatched shapes before anything reaches the library, and fails
loudly (no fallback) when the library is missing."""
import pytest
import torch

import bit_weight_only_g128_gb300 as w4
from bit_weight_only_g128_gb300 import build as wbuild


@pytest.fixture(scope="module")
def pw():
    wbuild.build()
    # a packed weight whose buffers live on the host: never handed to a kernel
    K, N, g = 256, 32, 128
    wb, sb, zb = w4.packed_sizes(K, N, g)
    return w4.PackedWeight(torch.zeros(wb // 4, dtype=torch.int32),
                           torch.zeros(sb // 2, dtype=torch.float16),
                           torch.zeros(zb // 4, dtype=torch.int32), K, N, g)


def test_packed_weight_bytes(pw):
    assert pw.nbytes == 256 * 32 // 2 + 2 * 2 * 32 + 2 * 32 // 2


def test_gemm_rejects_host_tensors_and_bad_shapes(pw):
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.gemm(torch.zeros((2, 256), dtype=torch.float16), pw)
    with pytest.raises(ValueError, match="K=128"):
        w4.gemm(torch.zeros((2, 128), dtype=torch.float16), pw)
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.gemm(torch.zeros((2, 256), dtype=torch.bfloat16), pw, silu_mul=True, a8=True)


def test_quantize_act_and_dequantize_checks(pw):
    with pytest.raises(ValueError, match="CUDA tensor"):
        w4.quantize_act(torch.zeros((2, 64), dtype=torch.float16))
    with pytest.raises(ValueError, match="float16 or bfloat16"):
        w4.dequantize(pw, dtype=torch.float32)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(w4, "_lib", None)
    monkeypatch.setattr(w4, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError, match="missing"):
        w4.lib()


def test_flag_values():
    assert (w4.STATIC_WEIGHTS, w4.SILU_MUL, w4.BF16, w4.ACT_A8) == (0x100, 0x200, 0x400, 0x800)
    assert set(w4._PATHS) == {"auto", "decode", "tensor", "decode-resident", "decode-streamk",
                              "tensor-pair"}
