"""Build ``libfa.so`` (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file;
the objects link into one shared library with the CUDA runtime linked
statically, so loading the library needs no GPU and no libcuda (the driver's
tensor-map encoder is looked up at run time).

    python -m numerics_tcgen05_tmem_gb300.build [--testhooks | --debug-bounds]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")
# Test-only build: FA_TEST_HOOKS compiles in the failure-injection hook and waits give up
# after 100 ms.  Never loaded by the binding, the benchmark or the smoke check.
LIB_TESTHOOKS = os.path.join(BUILD, "testhooks", "libfa_testhooks.so")
TESTHOOKS_FLAGS = ["-DFA_TEST_HOOKS=1", "-DFA_WAIT_TIMEOUT_NS=100000000ull"]
# Debug build: FA_DEBUG_BOUNDS checks the kernels' computed indices before each access and
# records the first violation in the status record (it never traps).  Loaded only by its test.
LIB_DEBUG_BOUNDS = os.path.join(BUILD, "debugbounds", "libfa_debugbounds.so")
DEBUG_BOUNDS_FLAGS = ["-DFA_DEBUG_BOUNDS=1"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libfa.so")
    return cand


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _needs_rebuild(extra_flags, lib=LIB, objdir=BUILD) -> bool:
    if not os.path.exists(lib):
        return True
    stamp = os.path.join(objdir, "flags.txt")
    if not os.path.exists(stamp) or open(stamp).read() != " ".join(extra_flags):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "fa.h")]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, testhooks: bool = False, debug_bounds: bool = False) -> str:
    extra = []
    lib, objdir = LIB, BUILD
    if testhooks and debug_bounds:
        raise ValueError("build one variant at a time")
    if testhooks:
        extra = extra + TESTHOOKS_FLAGS
        lib, objdir = LIB_TESTHOOKS, os.path.dirname(LIB_TESTHOOKS)
    if debug_bounds:
        extra = extra + DEBUG_BOUNDS_FLAGS
        lib, objdir = LIB_DEBUG_BOUNDS, os.path.dirname(LIB_DEBUG_BOUNDS)
    if not force and not _needs_rebuild(extra, lib, objdir):
        return lib
    nvcc = nvcc_path()
    os.makedirs(objdir, exist_ok=True)
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", CSRC,
                     "-I", os.path.join(HERE, "..", "include")] + extra

    def compile_one(src):
        obj = os.path.join(objdir, src[:-3] + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(os.path.join(objdir, "flags.txt"), "w") as f:
        f.write(" ".join(extra))
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--testhooks", action="store_true", help="build the failure-injection test library")
    ap.add_argument("--debug-bounds", action="store_true", help="build the index-checking debug library")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, testhooks=a.testhooks, debug_bounds=a.debug_bounds))


if __name__ == "__main__":
    main()
