"""Builds libqsa.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ compiles in parallel to an object file under
``_build/``; the objects link into ``block_sparse_gqa_qsa_gb300/libqsa.so``.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libqsa.so")
PEAKS_SRC = os.path.join(CSRC, "probes", "qsa_peaks.cu")
PEAKS_LIB = os.path.join(PKG, "libqsa_peaks.so")  # the benchmark's roofline probes (not part of the C ABI)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put /usr/local/cuda/bin on PATH")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "qsa.h")]


def _fresh(lib: str, deps) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(p) for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Builds libqsa.so (and libqsa_peaks.so) when a source is newer; returns the libqsa.so path."""
    peaks = None
    if force or not _fresh(PEAKS_LIB, [PEAKS_SRC]):
        tmp_p = PEAKS_LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-shared", PEAKS_SRC, "-o", tmp_p]
        peaks = (tmp_p, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    try:
        return _build_lib(force, verbose, extra_flags)
    finally:
        if peaks:
            out, _ = peaks[1].communicate()
            if peaks[1].returncode:
                print(out, file=sys.stderr)
                raise RuntimeError("nvcc failed for qsa_peaks.cu")
            os.replace(peaks[0], PEAKS_LIB)


def _build_lib(force: bool, verbose: bool, extra_flags) -> str:
    if not force and _fresh(LIB, _deps()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode):
            print(out, file=sys.stderr)
        if p.returncode:
            failed.append(os.path.basename(src))
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
