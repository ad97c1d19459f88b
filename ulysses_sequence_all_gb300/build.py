"""Compile libulysses.so in-tree for sm_103a (nvcc, one -gencode, sources compiled in parallel).

Usage: ``python -m ulysses_sequence_all_gb300.build`` or ``build_library()`` from Python.
Extra preprocessor definitions (engine tuning constants such as ``ULY_TMA_STAGES``) can be passed
through ``defines``; the default build uses the values in the sources.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBRARY = os.path.join(PKG, "libulysses.so")
SOURCES = ["api.cu", "relayout.cu", "fused_qk.cu", "fused_qk_tensor.cu", "fused_qk_bwd.cu",
           "plan.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _compile(src: str, obj: str, defines: dict, verbose_ptxas: bool) -> str:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
           "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd.insert(1, "-x=cu")
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    for k, v in defines.items():
        cmd.append(f"-D{k}={v}")
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{proc.stderr}")
    return proc.stderr


def build_library(out: str = LIBRARY, defines: dict | None = None, verbose_ptxas: bool = False,
                  build_dir: str | None = None) -> str:
    defines = defines or {}
    build_dir = build_dir or os.path.join(PKG, "_build")
    os.makedirs(build_dir, exist_ok=True)
    objs = [os.path.join(build_dir, os.path.splitext(s)[0] + ".o") for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        logs = list(pool.map(lambda so: _compile(so[0], so[1], defines, verbose_ptxas),
                             zip(SOURCES, objs)))
    if verbose_ptxas:
        for log in logs:
            if log:
                sys.stderr.write(log)
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"link failed:\n{proc.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build_library(verbose_ptxas="-v" in sys.argv))
