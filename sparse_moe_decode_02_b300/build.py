"""Build libflint.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m sparse_moe_decode_02_b300.build [--force]
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libflint.so")
SRC_MAIN = os.path.join(HERE, "csrc", "flint_all.cu")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "--shared", "-Xcompiler", "-fPIC",
    "-Xptxas", "-warn-spills",
]


def _sources():
    return (glob.glob(os.path.join(HERE, "csrc", "*.cu")) +
            glob.glob(os.path.join(HERE, "csrc", "*.cuh")) +
            glob.glob(os.path.join(HERE, "csrc", "*.h")) +
            [os.path.join(ROOT, "include", "flint.h")])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc] + NVCC_FLAGS + ["-o", tmp, SRC_MAIN]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
