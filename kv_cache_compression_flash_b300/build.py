"""Builds libkvs.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "kvs.cu")
OUT = os.path.join(HERE, "libkvs.so")
# the bounds-checked build: every data-dependent index is checked (KVS_DEBUG),
# a failed check records KVS_ERR_BOUNDS and skips the access
OUT_DEBUG = os.path.join(HERE, "libkvs_debug.so")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def nvcc_command(out=OUT, extra=()):
    return [os.path.join(CUDA_HOME, "bin", "nvcc"),
            "-gencode", "arch=compute_103a,code=sm_103a",
            "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC", "-shared",
            "-I", os.path.join(ROOT, "include"),
            "-cudart", "shared",
            "-Xlinker", "-rpath=" + os.path.join(CUDA_HOME, "lib64"),
            *extra, "-o", out, SRC]


def build_library(verbose=False, force=False, debug=False) -> str:
    """Builds libkvs.so (or, with debug, the bounds-checked libkvs_debug.so) unless it is newer than every source."""
    out = OUT_DEBUG if debug else OUT
    srcs = [os.path.join(HERE, "csrc", f) for f in os.listdir(os.path.join(HERE, "csrc"))]
    srcs.append(os.path.join(ROOT, "include", "kvs.h"))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(os.path.getmtime(s) for s in srcs):
        return out
    extra = (("-DKVS_DEBUG",) if debug else ()) + (("-Xptxas", "-v") if verbose else ())
    cmd = nvcc_command(out=out, extra=extra)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stderr)
    return out


if __name__ == "__main__":
    build_library(verbose=True, force=True)
