"""Compile the CUDA library in-tree for sm_103a (nvcc, no cmake)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libspecverify_debug.so")  # range-checked build (-DSV_DEBUG)
SOURCES = [os.path.join(CSRC, f) for f in ("spec_verify.cu", "sv_kv.cu", "sv_budget.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("sv_device.cuh", "sv_draw.cuh", "sv_stream.cuh", "sv_rescan.cuh",
                                                  "sv_decide.cuh", "sv_topkp.cuh", "sv_topkp_ring.cuh",
                                                  "sv_check.cuh")] + [
    os.path.join(INCLUDE, "spec_verify.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_command(out: str = LIB_PATH, debug: bool = False) -> list[str]:
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    return [nvcc, *NVCC_FLAGS, *(["-DSV_DEBUG"] if debug else []), "-I", INCLUDE, *SOURCES, "-o", out]


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def start_build(force: bool = False, debug: bool = False):
    """Start nvcc in the background; returns the Popen (or None when already built).  debug: the
    range-checked library (libspecverify_debug.so) instead of the release one."""
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and up_to_date(path):
        return None
    tmp = path + f".tmp{os.getpid()}"
    proc = subprocess.Popen(nvcc_command(tmp, debug))
    proc._sv_tmp, proc._sv_path = tmp, path  # type: ignore[attr-defined]
    return proc


def finish_build(proc) -> str:
    if proc is None:
        return LIB_PATH
    if proc.wait() != 0:
        raise RuntimeError(f"nvcc failed building {os.path.basename(proc._sv_path)}")  # type: ignore[attr-defined]
    os.replace(proc._sv_tmp, proc._sv_path)  # type: ignore[attr-defined]
    return proc._sv_path  # type: ignore[attr-defined]


def build(force: bool = False) -> str:
    finish_build(start_build(force))
    return LIB_PATH


def build_debug(force: bool = False) -> str:
    """The range-checked library: every global-memory access of every kernel checked (-DSV_DEBUG)."""
    finish_build(start_build(force, debug=True))
    return DEBUG_LIB_PATH
