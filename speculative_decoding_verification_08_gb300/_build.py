"""Builds libspecverify.so in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "specverify.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "sv_device.cuh"), os.path.join(CSRC, "sv_tma.cuh"),
                     os.path.join(CSRC, "sv_item.cuh"), os.path.join(CSRC, "sv_alpha.cuh"),
                     os.path.join(CSRC, "sv_logits.cuh"), os.path.join(CSRC, "sv_debug.cuh"),
                     os.path.join(CSRC, "sv_trace.cuh"),
                     os.path.join(INCLUDE, "specverify.h")]
LIBRARY = os.path.join(PKG, "libspecverify.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(f) <= t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the CUDA library (a few seconds) unless it is up to date."""
    if not force and up_to_date():
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


def build_variant(out: str, defines) -> str:
    """Compiles the library with extra -D flags into `out`; the regular
    build is left as it is."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *defines, "-I", INCLUDE, "-o", tmp, *SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build_debug(out: str) -> str:
    """A debug build (SV_DEBUG=1): every call checks its input rows for
    negative, NaN or infinite values before its kernels and reports them as
    SV_STATUS_BAD_VALUE."""
    return build_variant(out, ["-DSV_DEBUG=1"])


def build_trace(out: str) -> str:
    """A trace build (SV_TRACE=1): the item kernel records a timeline that
    sv_trace_read returns."""
    return build_variant(out, ["-DSV_TRACE=1"])
