"""Builds libw4a16.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu file compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically. Rebuilds only when a
source or header is newer than the library.

Two variants share the sources:
  ""           libw4a16.so, the library;
  "testhooks"  libw4a16_testhooks.so, the same code compiled with
               -DW4A16_TEST_HOOKS for the failure-path tests: its bounded
               waits take a limit the test sets and its TMA producers can be
               told to stop issuing copies (see csrc/internal.cuh).
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
VARIANTS = {"": [], "testhooks": ["-DW4A16_TEST_HOOKS"]}
LIB = os.path.join(PKG, "libw4a16.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def lib_path(variant: str = "") -> str:
    return os.path.join(PKG, f"libw4a16_{variant}.so" if variant else "libw4a16.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [
        os.path.abspath(__file__)]


def up_to_date(variant: str = "") -> bool:
    lib = lib_path(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build_variants(variants=("", "testhooks"), force: bool = False, verbose: bool = False, extra_flags=()):
    """Builds the given variants (compiling all their objects in one parallel pass)."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if not todo:
        return [lib_path(v) for v in variants]
    jobs = []
    for v in todo:
        out = os.path.join(BUILD, v or "lib")
        os.makedirs(out, exist_ok=True)
        for src in sources():
            jobs.append((v, src, os.path.join(out, os.path.basename(src)[:-3] + ".o")))

    def compile_one(job):
        v, src, obj = job
        cmd = [NVCC, *ARCH, *FLAGS, *VARIANTS[v], *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({v or 'lib'}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return job

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        done = list(ex.map(compile_one, jobs))
    for v in todo:
        objs = [obj for vv, _, obj in done if vv == v]
        lib = lib_path(v)
        tmp = lib + f".{os.getpid()}.tmp"
        r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed ({v or 'lib'}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return [lib_path(v) for v in variants]


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Builds one variant (the library by default) and returns its path."""
    return build_variants((variant,), force=force, verbose=verbose, extra_flags=extra_flags)[0]


if __name__ == "__main__":
    import sys
    print(build_variants(force="--force" in sys.argv, verbose=True))
