"""Build libdbf.so (all CUDA kernels and the C ABI) in-tree for sm_103a.

Usage: python -m double_binary_rank_packed_b300.build [--force] [--debug]
(--debug builds libdbf_debug.so, the library with the kernels' bounds checks)
Needs nvcc (CUDA 13) on PATH or under /usr/local/cuda/bin; no GPU is needed
to compile.
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libdbf.so")
# the debug build (bounds checks in the kernels, see in_range in csrc/common.cuh)
LIB_DEBUG = os.path.join(HERE, "libdbf_debug.so")
SOURCES = ["dbf_api.cu", "decode.cu", "decode_rs.cu", "prefill.cu", "misc.cu", "noalloc.cu", "factorize.cu", "factorize_tc.cu"]
HEADERS = ["common.cuh", "decode_frag.cuh", "kernels.h", "factorize.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libdbf.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "dbf.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, debug: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Build libdbf.so (or, with debug=True, libdbf_debug.so: the same library with the kernels'
    bounds checks compiled in) unless it is newer than every source; return its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    nvcc = nvcc_path()
    flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-shared",
             "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + ARCH
    if debug:
        flags += ["-DDBF_DEBUG=1"]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    tmp = lib + ".tmp"
    cmd = [nvcc] + flags + [os.path.join(CSRC, s) for s in SOURCES] + ["-o", tmp]
    if verbose:
        print(" ".join(cmd))
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if ptxas_info or verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    args = ap.parse_args(argv)
    path = build(force=args.force, debug=args.debug, verbose=True, ptxas_info=args.ptxas_info)
    print(path)


if __name__ == "__main__":
    main()
