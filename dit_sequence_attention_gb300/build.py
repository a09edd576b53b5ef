"""Build step for libh3attn.so (sm_103a), run in-tree.

Each ``csrc/*.cu`` translation unit is compiled by its own nvcc process (in
parallel), then linked into ``dit_sequence_attention_gb300/libh3attn.so``
with the CUDA runtime linked statically, so the library loads on a machine
without a GPU driver (the driver is looked up only when a call needs it).

``build(debug=True)`` makes ``libh3attn_debug.so`` from the same sources with
``H3ATTN_DEBUG_CHECKS=1``: every kernel checks each computed global index
before the access and reports a failed check through the device status word
(H3ATTN_ERR_DEVICE_BOUNDS) instead of touching memory outside its buffers.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libh3attn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libh3attn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libh3attn.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile every CUDA translation unit for sm_103a and link libh3attn.so
    (``debug=True``: libh3attn_debug.so, with the device index checks)."""
    lib = LIB_DEBUG if debug else LIB
    bdir = BUILD_DEBUG if debug else BUILD
    if not force and up_to_date(debug):
        return lib
    os.makedirs(bdir, exist_ok=True)
    exe = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DH3ATTN_DEBUG_CHECKS=1"] if debug else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
