"""Builds the CUDA library in-tree: bit_quantized_lora_double_b300/libqlora_b300.so.

nvcc compiles csrc/qlora_lib.cu (which includes every kernel) for sm_103a
only, with the CUDA runtime linked statically so the library loads on a
machine without a GPU (calls then fail with a CUDA error instead).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libqlora_b300.so")
# diagnostic build: the same library with the fused GEMM recording per-step
# timestamps of one CTA pair (see profile_case.py --stamps)
STAMPS_LIB = os.path.join(PKG, "libqlora_b300_stamps.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2", "-shared",
    "--expt-relaxed-constexpr",
    "-I", os.path.join(ROOT, "include"),
    "-I", CSRC,
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "qlora.h")])


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, stamps: bool = False) -> str:
    lib = STAMPS_LIB if stamps else LIB
    if not force and not needs_build(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *FLAGS, *(["-DQLORA_GEMM_STAMPS"] if stamps else []), *(["-Xptxas", "-v"] if ptxas_v else []),
           "-o", tmp, os.path.join(CSRC, "qlora_lib.cu")]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose or ptxas_v:
        sys.stderr.write(r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)
