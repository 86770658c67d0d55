"""Build libtpmlp.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtpmlp.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpmlp.so")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(INCLUDE, "tpmlp.h"), __file__])


def source_hash(extra_flags=()) -> str:
    """16 hex digits of SHA-256 over the library's sources (csrc/, include/tpmlp.h, by
    relative path and content) and the compile flags. Built into the library
    (tpmlp_build_id), so that a measurement recorded against one build of the kernels can be
    told apart from another build's."""
    h = hashlib.sha256()
    files = sorted(sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
                   glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(INCLUDE, "tpmlp.h")])
    for path in files:
        h.update(os.path.relpath(path, ROOT).encode())
        h.update(b"\0")
        with open(path, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join([*ARCH_FLAGS, "-O3", *extra_flags]).encode())
    return h.hexdigest()[:16]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = None) -> str:
    """Compile every .cu under csrc/ into one shared library (a few seconds per kernel
    instantiation). Returns the library path. `out` + `extra_flags` build a variant (for
    instance a test build with a planted pipeline stall) at another path."""
    lib = out or LIB
    if out is None and not force and not stale():
        return LIB
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", INCLUDE,
           "-I", CSRC, "-DTPMLP_BUILD", f'-DTPMLP_SOURCE_HASH="{source_hash(extra_flags)}"',
           *extra_flags, *sources(), "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib
