"""Builds libgdn.so in-tree with nvcc for sm_103a (B300), and its debug build
libgdn_debug.so (-DGDN_DEBUG=1: every kernel checks its scratch offsets against the
host layout's region extents and reports GDN_ERR_BOUNDS instead of touching
memory outside them)."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(PKG, "libgdn.so")
LIB_DEBUG = os.path.join(PKG, "libgdn_debug.so")
CSRC = os.path.join(PKG, "csrc")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    newest = max(os.path.getmtime(p) for p in sources() + glob.glob(os.path.join(CSRC, "*.h"))
                 + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(PKG, "..", "include", "gdn.h")])
    return newest > os.path.getmtime(lib)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compiles csrc/*.cu into libgdn.so (libgdn_debug.so with ``debug``) next to
    this file; returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + ".tmp"
    cmd = [NVCC, *FLAGS, *(["-DGDN_DEBUG=1"] if debug else []), *(["-Xptxas", "-v"] if verbose else []), "-o", tmp,
           *sources()]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, lib)
    return lib


def ensure_built(debug: bool = False) -> str:
    """Builds only when the library is missing (used by tests on a GPU machine, where the
    snapshot already carries the library built here)."""
    lib = LIB_DEBUG if debug else LIB
    if os.path.exists(lib) and os.environ.get("GDN_FORCE_REBUILD") != "1":
        return lib
    return build(force=True, debug=debug)
