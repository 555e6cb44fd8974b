"""Build libgbattn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel, then one
link step produces ``attention_forward_09_gb300/libgbattn.so``.  The library
links the CUDA runtime dynamically and resolves ``cuTensorMapEncodeTiled``
through the runtime's driver entry-point query, so it does not link libcuda.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgbattn.so")
SOURCES = ["api.cpp", "prefill.cu", "decode.cu", "noalloc.cu", "cache_write.cu", "masks.cu", "vsa_layout.cpp", "vsa.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libgbattn.so")
    return cand


def cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _compile(nv: str, src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, src + ".o")
    cmd = [nv, "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", os.path.join(os.path.dirname(PKG), "include")] + ARCH
    if src.endswith(".cu") and verbose:
        cmd += ["-Xptxas", "-v"]
    if src.endswith(".cpp"):
        cmd = [nv, "-x", "cu"] + cmd[1:]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link; returns the path of libgbattn.so.  Skips the work
    when the library is newer than every source (unless ``force``)."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES] + [
        os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))
    ] + [os.path.join(os.path.dirname(PKG), "include", "gbattn.h"), __file__]
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(s) for s in srcs)
        if os.path.getmtime(LIB) >= newest:
            return LIB
    nv = nvcc()
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nv, s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nv, "-shared", "-o", tmp] + objs + ARCH + [
        "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib_dir(nv)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
