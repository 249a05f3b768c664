"""Build step of the C-ABI library ``libspecverify.so`` (sm_103a).

Two translation units (the verify step, and its vocabulary-sharded form),
one ``-gencode``, compiled in-tree next to this file with ``nvcc -shared``.  Rebuilds only when a source or the header is newer
than the library.
"""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libspecverify.so")
SOURCES = [os.path.join(CSRC, "spec_verify.cu"), os.path.join(CSRC, "sv_shard.cu")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libspecverify.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libspecverify.so if needed; returns its path."""
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(f) <= t for f in _deps()):
            return LIB
    cmd = [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-Xptxas", "-v" if verbose else "-O3",
           "-I", INCLUDE, "-I", CSRC, *SOURCES, "-o", LIB + ".tmp", "-lcudart"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
