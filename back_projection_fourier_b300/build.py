"""Build libtp.so in-tree with nvcc for sm_103a (B300).

    python -m back_projection_fourier_b300.build [--verbose]

The library is written next to this file so that it travels with the source tree.
"""
from __future__ import annotations

import os
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
LIB = PKG / "libtp.so"
INCLUDE = PKG.parent / "include"
SOURCES = ["kernels.cu", "pad.cu", "tp_abi.cu", "no_alloc.cu"]
# microbenchmarks of the on-chip units (include/tp_peaks.h), a library of their own
PEAKS_LIB = PKG / "libtp_peaks.so"
PEAKS_SOURCES = ["peaks.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        [INCLUDE / "tp.h"]


def stale() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _inputs())


def _compile(lib: Path, sources, verbose: bool) -> None:
    tmp = lib.with_name(f"{lib.name}.{os.getpid()}")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", str(INCLUDE), "-o", str(tmp)]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [str(CSRC / s) for s in sources]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile every CUDA source of the package: libtp.so and the microbenchmarks'
    libtp_peaks.so (each a no-op when up to date)."""
    if force or stale():
        _compile(LIB, SOURCES, verbose)
    peak_inputs = [CSRC / s for s in PEAKS_SOURCES] + [INCLUDE / "tp_peaks.h"]
    if force or not PEAKS_LIB.exists() or any(
            p.stat().st_mtime > PEAKS_LIB.stat().st_mtime for p in peak_inputs):
        _compile(PEAKS_LIB, PEAKS_SOURCES, verbose)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB)
