"""Builds libherald.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel, then linked into one
shared library with a C ABI (include/herald.h).  No CMake, no torch
extension machinery: the library depends only on the CUDA runtime.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libherald.so")
# the debug build: the same sources with -DHERALD_DEBUG (device checks of
# indices and counts, read through herald_debug_status)
DEBUG_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libherald.so")
SOURCES = ["herald_api.cu", "select_kernels.cu", "tc_kernels.cu", "attn_flash.cu",
           "move_kernels.cu", "block_select.cu", "herald_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(os.path.dirname(HERE), "include", "herald.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          debug: bool = False) -> str:
    out_dir, lib = (DEBUG_DIR, DEBUG_LIB) if debug else (OUT_DIR, LIB)
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    cc = nvcc()
    flags = FLAGS + (["-DHERALD_DEBUG"] if debug else []) + (extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
