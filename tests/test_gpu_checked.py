"""The bounds-checked build on the GPU.

The library is rebuilt with -DW4A16_CHECKED (every global and shared-memory
access of every kernel tested against its buffer's extent first; an access
outside sets bit 64 of the device error word and is skipped) and the parity
suites of the small shapes run against it in a child process: each test
reads the device error word after its calls (w4a16_device_status), so a
single out-of-bounds access anywhere fails it. The caller-owned workspaces
of these suites are checked by their own tests (zero-filled flag areas, Y
inside sentinel padding); here the workspace is additionally given canary
bytes past the size the library asked for, which must stay untouched.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bit_weight_only_g128_gb300 import build as wbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_prep.py", "tests/test_gpu_gemm.py", "tests/test_gpu_tensor.py",
          "tests/test_gpu_silu.py", "tests/test_gpu_bf16.py", "tests/test_gpu_a8.py",
          "tests/test_gpu_flags.py"]


def _child_env(lib):
    env = dict(os.environ)
    env["W4A16_LIBRARY"] = lib
    env.pop("W4A16_MARGINS_FILE", None)
    return env


def test_parity_suites_pass_in_the_checked_build():
    lib = wbuild.build(checked=True)
    res = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-q", "-x", "-m", "gpu",
                          "-p", "no:cacheprovider"],
                         cwd=ROOT, env=_child_env(lib), capture_output=True, text=True, timeout=1800)
    tail = "\n".join((res.stdout + res.stderr).splitlines()[-30:])
    assert res.returncode == 0, tail
    assert " passed" in tail and " failed" not in tail, tail


CANARY_SCRIPT = r"""
import sys
import numpy as np, torch
import bit_weight_only_g128_gb300 as w4
assert w4.LIB_PATH.endswith("libw4a16_checked.so"), w4.LIB_PATH
torch.manual_seed(0)
cases = [(8, 1024, 384, 128, "decode-streamk", 0), (48, 2048, 400, 128, "tensor", 3),
         (300, 1024, 512, 128, "tensor", 2), (600, 1024, 768, 128, "tensor-pair", 0),
         (5, 2048, 512, 2048, "decode", 0)]
for M, K, N, g, path, parts in cases:
    W = torch.randn(K, N, device="cuda") * 0.02
    pw = w4.quantize_pack(W, g)
    A = torch.randn(M, K, device="cuda").half()
    need = w4.workspace_size(M, N, K, g, path, parts)
    pad = 4096
    buf = torch.zeros(need + pad, dtype=torch.uint8, device="cuda")
    buf[need:] = 0xA5
    Y = w4.gemm(A, pw, path=path, parts=parts, workspace=buf[:need] if need else None)
    w4.device_status()
    assert bool((buf[need:] == 0xA5).all()), (M, K, N, path, "wrote past the workspace")
    ref = A.float() @ w4.dequantize(pw).float()
    err = (Y.float() - ref).abs().max().item()
    assert err <= 2 ** -9 * (A.float().abs() @ w4.dequantize(pw).float().abs()).max().item() + 1e-3, (M, K, N, path, err)
print("canaries ok")
"""


def test_workspace_canaries_in_the_checked_build():
    lib = wbuild.build(checked=True)
    res = subprocess.run([sys.executable, "-c", CANARY_SCRIPT], cwd=ROOT, env=_child_env(lib),
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "canaries ok" in res.stdout, (res.stdout + res.stderr)[-3000:]
