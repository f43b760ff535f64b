"""Builds libspecverify.so (the C-ABI CUDA library) in-tree for sm_103a.

Usage: ``python -m speculative_decoding_verification_44_gb300.build [-v]``.
No PyTorch involvement: one nvcc invocation, host code C++17, device code
sm_103a only.
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
LIB_NAME = "libspecverify.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["spec_verify.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify.so")


def nvcc_command(out: str = LIB_PATH, extra: list[str] | None = None) -> list[str]:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
            "-I", INCLUDE, "-I", CSRC, "-o", out,
            *[os.path.join(CSRC, s) for s in SOURCES], *(extra or [])]


def sources_newer_than(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(d) > t for d in deps) or os.path.getmtime(__file__) > t


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    if not force and not sources_newer_than(LIB_PATH):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else None)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force=True))
