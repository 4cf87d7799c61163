"""Build libtsa.so (and its debug build libtsa_debug.so) in-tree with nvcc for
sm_103a (B300).

Usage: python -m fixed_state_recurrence_phi_b300.build  [--force] [--debug | --all]
The libraries are placed next to this file; the Python binding loads
libtsa.so, or libtsa_debug.so when TSA_DEBUG=1 is set in the environment.
Each translation unit is compiled on its own (in parallel) into _build/, then
linked.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libtsa.so")
LIB_DEBUG = os.path.join(HERE, "libtsa_debug.so")
OBJ_DIR = os.path.join(HERE, "_build")
SOURCES = ["tsa_abi.cu", "prefill_tc.cu", "prefill_tc32.cu", "prefill_pair.cu", "prefill_short.cu", "tsa_noalloc.cu"]
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-std=c++17", "-O3", "-lineinfo",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]
# the debug build: device-side checks before each TMEM, shared-memory operand,
# TMA and state access (csrc/debug_check.cuh)
DEBUG_FLAGS = ["-DTSA_DEBUG"]


def _inputs():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(os.path.dirname(HERE), "include", "tsa.h"))
    return out


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(nvcc: str, src: str, obj: str, flags: list[str], verbose: bool) -> None:
    cmd = [nvcc, *NVCC_FLAGS, *flags, "-c", "-o", obj, os.path.join(CSRC, src)]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True, cwd=CSRC)


def _build_many(variants: list[bool], verbose: bool) -> None:
    """Compile every translation unit of each variant (False = release,
    True = debug) in parallel, then link each library."""
    nvcc = os.environ.get("NVCC", "nvcc")
    os.makedirs(OBJ_DIR, exist_ok=True)
    jobs = []
    for debug in variants:
        tag = "dbg" if debug else "rel"
        for src in SOURCES:
            obj = os.path.join(OBJ_DIR, f"{os.path.splitext(src)[0]}.{tag}.o")
            jobs.append((src, obj, DEBUG_FLAGS if debug else []))
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for f in [ex.submit(_compile, nvcc, s, o, fl, verbose) for s, o, fl in jobs]:
            f.result()
    for debug in variants:
        tag = "dbg" if debug else "rel"
        lib = LIB_DEBUG if debug else LIB
        objs = [os.path.join(OBJ_DIR, f"{os.path.splitext(s)[0]}.{tag}.o") for s in SOURCES]
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", lib + ".tmp", *objs]
        if verbose:
            print(" ".join(cmd))
        subprocess.run(cmd, check=True, cwd=CSRC)
        os.replace(lib + ".tmp", lib)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build the release library (or, with debug=True, the debug library) if
    any source is newer. Returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if force or not up_to_date(debug):
        _build_many([debug], verbose)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> list[str]:
    """Build both libraries (their translation units compile in parallel)."""
    variants = [d for d in (False, True) if force or not up_to_date(d)]
    if variants:
        _build_many(variants, verbose)
    return [LIB, LIB_DEBUG]


if __name__ == "__main__":
    force = "--force" in sys.argv
    if "--all" in sys.argv:
        print(build_all(force=force, verbose=True))
    else:
        print(build(force=force, verbose=True, debug="--debug" in sys.argv))
