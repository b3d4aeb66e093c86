"""Build step of the CUDA library: one nvcc invocation, in-tree.

Produces ``libcfgstep.so`` next to this file from ``csrc/cfgstep.cu`` (the
kernels and the step entry points) and ``csrc/cfgstep_host.cpp`` (host tables
and sampler loops) for sm_103a (B300).  Only the ``extern "C"`` entry points declared in
``include/cfgstep.h`` are exported (hidden visibility for everything else).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG_DIR = Path(__file__).resolve().parent
REPO_DIR = PKG_DIR.parent
SRC = PKG_DIR / "csrc" / "cfgstep.cu"
SOURCES = [SRC, PKG_DIR / "csrc" / "cfgstep_host.cpp"]
INTERNAL = PKG_DIR / "csrc" / "cfgstep_internal.h"
NOISE = PKG_DIR / "csrc" / "cfg_noise.cuh"
HEADER = REPO_DIR / "include" / "cfgstep.h"
LIB = PKG_DIR / "libcfgstep.so"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def nvcc_command(out: Path = LIB, extra: list[str] | None = None) -> list[str]:
    cuda_lib = Path(nvcc_path()).resolve().parent.parent / "lib64"
    return [
        nvcc_path(), *ARCH_FLAGS, "-lineinfo", "-O3", "-std=c++17",
        "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
        "-cudart", "shared", f"-Xlinker=-rpath,{cuda_lib}",
        "-I", str(HEADER.parent),
        *(extra or []),
        "-o", str(out), *map(str, SOURCES),
    ]


def needs_build() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in (*SOURCES, INTERNAL, NOISE, HEADER, Path(__file__)))


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile the library if it is missing or older than its sources; return its path."""
    if not force and not needs_build():
        return LIB
    cmd = nvcc_command()
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    tmp = LIB.with_suffix(".so.tmp")
    cmd[cmd.index("-o") + 1] = str(tmp)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout, res.stderr, file=sys.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
