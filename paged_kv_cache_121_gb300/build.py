"""Build libpa.so (the C-ABI library) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc (one -gencode, no
cmake); the objects are linked into ``paged_kv_cache_121_gb300/_build/libpa.so``.
Run ``python -m paged_kv_cache_121_gb300.build`` or call :func:`build`.
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
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libpa.so")

SOURCES = ["api.cu", "decode_mma.cu", "decode_balanced.cu", "prefix_mma.cu", "prefix_tc.cu", "decode_simt.cu", "cache_ops.cu",
           "decode_static.cu", "health.cu", "block_manager.cpp"]
HEADERS = ["device_common.cuh", "mma_tile.cuh", "tcgen05.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa")
    return path


def _flags(src: str):
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden"]
    if src.endswith(".cu"):
        return ARCH + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-v"] + common
    return common


def _compile(src: str) -> tuple:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + _flags(src) + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "pa.h"),
                                                                  os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpa.so if any source changed; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    failed = [r for r in results if r[2] != 0]
    for src, _, _, log in results:
        if verbose or any(f[0] == src for f in failed):
            sys.stderr.write(f"--- {src}\n{log}\n")
    if failed:
        raise RuntimeError("libpa build failed: " + ", ".join(f[0] for f in failed))
    tmp = LIB_PATH + ".tmp%d" % os.getpid()
    link = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [r[1] for r in results]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("libpa link failed")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
