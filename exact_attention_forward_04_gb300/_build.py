"""Build the CUDA library in-tree with nvcc for sm_103a.

    python -m exact_attention_forward_04_gb300._build [--force]

Output: exact_attention_forward_04_gb300/_lib/libfa_fwd.so (git-ignored), and
the ptxas resource report (registers, spills, shared memory) beside it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libfa_fwd.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _sources():
    files = []
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                files.append(os.path.join(d, name))
    return files


def _nvcc():
    cand = shutil.which("nvcc")
    if cand:
        return cand
    for p in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(p):
            return p
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def needs_build() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa_fwd.so if it is missing or older than its sources."""
    if not force and not needs_build():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        _nvcc(), ARCH, "-std=c++17", "-O3", "-lineinfo", "-shared",
        "-Xcompiler", "-fPIC", "-Xptxas", "-v",
        "-I", INCLUDE, "-I", CSRC,
        "-o", tmp, os.path.join(CSRC, "fa_fwd.cu"),
    ]
    res = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(OUT_DIR, "ptxas_report.txt"), "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(res.stderr)
    return LIB_PATH


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose=True)
    print(path)
