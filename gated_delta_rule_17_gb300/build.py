"""Builds the CUDA library in-tree: ``_lib/libgdn_gb300.so`` for sm_103a.

One translation unit (``csrc/gdn_api.cu``, which includes the kernels), so a
build takes a few seconds on either the x86 build host or the Arm GPU host.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "gdn_api.cu")
DEPS = [os.path.join(HERE, "csrc", f) for f in ("gdn_api.cu", "gdn_common.cuh", "gdn_prefill_kernel.cuh", "gdn_decode_kernel.cuh",
                                                           "gdn_wy_kernel.cuh", "gdn_bwd_common.cuh", "gdn_bwd_dstates_tc.cuh", "gdn_bwd_grads_tc.cuh",
                                                           "tc.cuh")] + [
    os.path.join(os.path.dirname(HERE), "include", "gdn_prefill.h")]
OUT_DIR = os.path.join(HERE, "_lib")
OUT = os.path.join(OUT_DIR, "libgdn_gb300.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(os.path.dirname(HERE), "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(OUT):
        newest = max(os.path.getmtime(d) for d in DEPS)
        if os.path.getmtime(OUT) >= newest:
            return OUT
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-o", tmp, SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True, verbose=True))
