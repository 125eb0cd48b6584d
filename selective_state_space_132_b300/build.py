"""Build libssm.so in-tree with nvcc for sm_103a (B300).

    python -m selective_state_space_132_b300.build [--force] [--verbose] [--debug-bounds]

The library is placed next to this file so that it travels with the source
tree; it links the CUDA runtime statically and exports only the C ABI of
include/ssm.h.  --debug-bounds builds libssm_debug.so instead: the same library
compiled with SSM_DEBUG_BOUNDS=1, whose kernels check the indices of their global
writes and TMA coordinates and record SSM_ERR_BOUNDS in the status word (skipping the
access) instead of faulting.  Load it with SSM_LIBRARY=<path>.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libssm.so")
LIB_DEBUG = os.path.join(HERE, "libssm_debug.so")
HEADER = os.path.join(ROOT, "include", "ssm.h")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    files = sources() + [HEADER]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return files


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug_bounds: bool = False) -> str:
    lib = LIB_DEBUG if debug_bounds else LIB
    if not force and up_to_date(lib):
        return lib
    objdir = os.path.join(ROOT, "_build_debug" if debug_bounds else "_build")
    os.makedirs(objdir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                    "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]
    if verbose:
        flags += ["-Xptxas", "-v"]
    flags += list(extra_flags or [])
    if debug_bounds:
        flags += ["-DSSM_DEBUG_BOUNDS=1"]
    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc()] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    # the translation units are independent: compile them side by side
    objs = []
    workers = max(1, min(len(sources()), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as pool:
        for src, obj, r in pool.map(compile_one, sources()):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
            objs.append(obj)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug_bounds=a.debug_bounds))
