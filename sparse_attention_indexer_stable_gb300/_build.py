"""Builds the CUDA library in-tree: csrc/*.cu -> _build/libdcp_topk.so (sm_103a).

Plain nvcc, one translation unit, no CMake; host code has no
architecture-specific flags so the same source builds on x86_64 and aarch64.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libdcp_topk.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


# The race-check build: the same library compiled with -DDCP_DEBUG_POISON
# (odd warps delayed after every barrier, shared state overwritten with
# garbage before every reset, indices from shared state clamped), for the
# barrier tests only; it exports the same C ABI.
POISON_LIB_PATH = os.path.join(OUT_DIR, "libdcp_topk_racecheck.so")
POISON_FLAGS = ("-DDCP_DEBUG_POISON",)


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, extra_flags=(), path: str = LIB_PATH) -> str:
    """Compile the library if missing or older than its sources; returns its path."""
    if not force and not is_stale(path):
        return path
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = path + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "--shared",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-o", tmp, *sources(), *extra_flags]
    subprocess.check_call(cmd)
    os.replace(tmp, path)
    return path


def build_race_check(force: bool = False) -> str:
    """The race-check build (see POISON_LIB_PATH); returns its path."""
    return build(force, POISON_FLAGS, POISON_LIB_PATH)
