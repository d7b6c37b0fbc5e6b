"""Build liblora_punica.so (sm_103a) in-tree with nvcc.

Usage: ``python -m expand_gemm_gb300.build [--force] [--debug]``.  Every
``.cu`` file under ``csrc/`` is compiled in parallel to ``_build/`` and
linked into ``expand_gemm_gb300/liblora_punica.so``.  Only the
``extern "C"`` entry points declared in ``include/lora_punica.h`` are
exported (hidden default visibility).  Works without a GPU (nvcc
cross-compiles).

``--debug`` builds ``liblora_punica_debug.so`` (objects in
``_build/debug/``) with ``LORA_PUNICA_DEBUG_CHECKS`` defined: every kernel
range-checks the LoRA ids, token indices and segment bounds it takes from
the metadata and reports a bad one in bit 29 of the error word instead of
using it.  Load it by setting ``LORA_PUNICA_LIBRARY`` to its path before
the first library call.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "liblora_punica.so")
DEBUG_LIB = os.path.join(PKG, "liblora_punica_debug.so")
DEBUG_FLAGS = ["-DLORA_PUNICA_DEBUG_CHECKS"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-I", INCLUDE, "-I", CSRC,
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and not is_stale(lib):
        return lib
    nvcc = _nvcc()
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    flags = list(extra_flags) + (DEBUG_FLAGS if debug else [])
    os.makedirs(bdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + flags + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-X")]
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, extra_flags=extra,
                debug="--debug" in sys.argv))
