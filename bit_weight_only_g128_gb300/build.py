"""Build the CUDA library in-tree: csrc/*.cu -> _build/libw4a16.so (sm_103a).

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library against the shared CUDA runtime (the one PyTorch loads).
``build(checked=True)`` builds the bounds-checked variant instead
(-DW4A16_CHECKED, _build/checked/libw4a16_checked.so): every global and
shared-memory access of its kernels is tested against its buffer first, and
an access outside sets a bit of the device error word instead of running.
Load it by setting W4A16_LIBRARY to its path before the binding loads the
library. Running ``python -m bit_weight_only_g128_gb300.build [--checked]``
builds by hand.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libw4a16.so")
BUILD_CHECKED = os.path.join(BUILD, "checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libw4a16_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin/ on PATH)")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, obj: str, extra) -> str:
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libw4a16.so (with
    `checked`, the bounds-checked libw4a16_checked.so); returns its path."""
    out_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in sources]
    extra = list(extra_flags) + (["-DW4A16_CHECKED"] if checked else []) + (["-Xptxas", "-v"] if verbose else [])
    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], extra), zip(sources, objs)))
    if verbose:
        for src, log in zip(sources, logs):
            if log.strip():
                print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
