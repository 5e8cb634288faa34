"""Compile the CUDA library in-tree for sm_103a (nvcc, no cmake)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
SOURCES = [os.path.join(CSRC, f) for f in ("spec_verify.cu", "sv_kv.cu", "sv_budget.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("sv_device.cuh", "sv_draw.cuh", "sv_stream.cuh", "sv_rescan.cuh", "sv_decide.cuh", "sv_topkp.cuh")] + [
    os.path.join(INCLUDE, "spec_verify.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc_command(out: str = LIB_PATH) -> list[str]:
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    return [nvcc, *NVCC_FLAGS, "-I", INCLUDE, *SOURCES, "-o", out]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def start_build(force: bool = False):
    """Start nvcc in the background; returns the Popen (or None when already built)."""
    if not force and up_to_date():
        return None
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    proc = subprocess.Popen(nvcc_command(tmp))
    proc._sv_tmp = tmp  # type: ignore[attr-defined]
    return proc


def finish_build(proc) -> str:
    if proc is not None:
        if proc.wait() != 0:
            raise RuntimeError("nvcc failed building libspecverify.so")
        os.replace(proc._sv_tmp, LIB_PATH)  # type: ignore[attr-defined]
    return LIB_PATH


def build(force: bool = False) -> str:
    return finish_build(start_build(force))
