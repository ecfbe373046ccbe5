"""Compile the CUDA library (libt2va.so) in-tree for sm_103a with nvcc."""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libt2va.so")
SOURCES = ["t2va_api.cu", "t2va_noise.cu", "t2va_objective.cu", "t2va_noalloc.cu", "t2va_w8a8.cu",
           "t2va_w8a8_tc.cu", "t2va_fused.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def command(out: str = LIB, extra=()) -> list:
    return ([nvcc(), "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xptxas", "-v",
             "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC, "-o", out]
            + [os.path.join(CSRC, s) for s in SOURCES] + list(extra))


def build(verbose: bool = False, force: bool = False) -> str:
    """Build libt2va.so if any source is newer than it; returns its path."""
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "t2va.h")]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(d) for d in deps):
            return LIB
    cmd = command()
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed building libt2va.so")
    return LIB


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)
