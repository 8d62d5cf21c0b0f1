"""Build step of the shard-step library: compiles csrc/ into libss.so with nvcc for sm_103a.

One translation unit per part of the ABI (host layout code; the fused step,
in two parts by the arrays' alignment; the reduce; the norm clip; the copies; shared host helpers), compiled in
parallel by nvcc and linked against the shared CUDA runtime so the library
shares the runtime instance of the process that loads it (e.g. PyTorch's).
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libss.so")

SOURCES = ["ss_layout.cpp", "ss_util.cu", "ss_step.cu", "ss_step_shift.cu", "ss_reduce.cu", "ss_norm.cu", "ss_copy.cu"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the shard-step library needs the CUDA toolkit to build")
    return exe


def build(verbose: bool = False) -> str:
    """Compile libss.so in place and return its path."""
    cmd = [nvcc(), "-std=c++17", "-O3", "-shared", "-lineinfo",
           "-gencode", "arch=compute_103a,code=sm_103a",
           "-fmad=false",                                  # every FMA in the update is explicit
           "-Xcompiler", "-fPIC,-ffp-contract=off",
           "-cudart", "shared", "--threads", str(len(SOURCES)),
           *[os.path.join(CSRC, s) for s in SOURCES], "-o", LIB]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if verbose and (p.stdout or p.stderr):
        print(p.stdout, p.stderr)
    if p.returncode != 0:
        raise RuntimeError(f"libss build failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
