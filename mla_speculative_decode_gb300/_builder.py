"""Builds libverifyattn.so (the CUDA kernels and the C ABI) for sm_103a in-tree.

Each .cu file is compiled by nvcc in parallel and linked into one shared
library under ``_build/``.  No cmake, no torch extension machinery: the
library exports only the C functions declared in include/verify_attn.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libverifyattn.so")
# The test build: the same sources with VA_TEST_HOOKS, which adds the
# producer gate declared in include/verify_attn_testhooks.h (used only by the
# bounded-wait test; the product library never contains it).
TESTHOOKS_LIB = os.path.join(OUT_DIR, "libverifyattn_testhooks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libverifyattn.so")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          testhooks: bool = False) -> str:
    """Builds libverifyattn.so, or with testhooks=True the test build
    libverifyattn_testhooks.so; returns the library's path."""
    lib = TESTHOOKS_LIB if testhooks else LIB
    if not force and up_to_date(lib):
        return lib
    obj_dir = os.path.join(OUT_DIR, "testhooks") if testhooks else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-I", CSRC,
                     "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr"]
    if testhooks:
        common += ["-DVA_TEST_HOOKS"]
    if ptxas_v:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_v:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcuda"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_v="--ptxas" in sys.argv, testhooks="--testhooks" in sys.argv))
