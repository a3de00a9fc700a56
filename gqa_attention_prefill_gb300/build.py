"""Compiles the CUDA library (libtsk_mha.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libtsk_mha.so")
SOURCES = [os.path.join(CSRC, "tsk_mha.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("attention.cuh", "attention_d128.cuh", "attention_fp8.cuh", "decode.cuh", "ptx.cuh", "schedule.cuh", "probe.cuh")] + [
    os.path.join(ROOT, "include", "tsk_mha.h")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def flags(verbose: bool = False):
    f = ["-std=c++17", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
         "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(ROOT, "include"),
         "-Xcompiler", "-fvisibility=hidden"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False, out: str | None = None,
          defines=(), host_flags=()) -> str:
    """Builds libtsk_mha.so (or `out`, with extra -D `defines` and host-compiler
    flags, always rebuilt)."""
    target = out or LIB
    if out is None and not defines and not host_flags and not force and not stale():
        return LIB
    tmp = target + f".tmp{os.getpid()}"
    hf = [x for f in host_flags for x in ("-Xcompiler", f)]
    cmd = [nvcc(), *flags(verbose), *[f"-D{d}" for d in defines], *hf, "-o", tmp, *SOURCES]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libtsk_mha.so")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, target)
    return target


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", action="store_true")
    ap.add_argument("--out")
    ap.add_argument("-D", action="append", default=[])
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.v, out=a.out, defines=a.D))
