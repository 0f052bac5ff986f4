"""Build the CUDA library in-tree: nvcc for sm_103a, one translation unit per
process, linked into lossless_entropy_coding_gb300/_build/libecc_gb300.so.
build(checked=True) builds the index-checked variant (-DECC_CHECKED: the
kernels test their shared- and global-memory indices, skip an access out of
range and report ECC_ERR_CHECK) into _build_checked/libecc_gb300_checked.so.

    python -m lossless_entropy_coding_gb300.build [--force] [--checked]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libecc_gb300.so")
CHECKED_DIR = os.path.join(HERE, "_build_checked")
CHECKED_LIB = os.path.join(CHECKED_DIR, "libecc_gb300_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "ecc.h"))
    return files


def _compile(src: str, nvcc: str, extra, out_dir: str = OUT_DIR) -> str:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           *extra, "-c", src, "-o", obj]
    subprocess.check_call(cmd)
    return obj


def build(force: bool = False, extra=(), checked: bool = False) -> str:
    out_dir, lib = (CHECKED_DIR, CHECKED_LIB) if checked else (OUT_DIR, LIB)
    flags = list(extra) + (["-DECC_CHECKED"] if checked else [])
    os.makedirs(out_dir, exist_ok=True)
    newest = max(os.path.getmtime(f) for f in _deps())
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(sources())) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc, flags, out_dir), sources()))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, checked="--checked" in sys.argv))
