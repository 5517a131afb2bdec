"""Builds libcp_attn.so in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library under ``_build/`` next to this file. A stamp of the sources and flags
avoids needless rebuilds.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcp_attn.so")
STAMP = os.path.join(BUILD, "stamp.txt")

SOURCES = ["api.cu", "plan.cpp", "step_fwd.cu", "step_bwd.cu", "hbm_kernels.cu",
           "noalloc.cu", "decode.cu", "fp8.cu"]
HEADERS = ["internal.h", "kernels.h", "ptx.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libcp_attn")
    return cand


def _digest(extra) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(ROOT, "include", "cp_attn.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(verbose: bool = False, extra_flags=(), force: bool = False) -> str:
    """Compile (if needed) and return the path of libcp_attn.so."""
    os.makedirs(BUILD, exist_ok=True)
    digest = _digest(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as f:
            if f.read().strip() == digest:
                return LIB
    nvcc = _nvcc()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".", "_") + ".o")
        objs.append(obj)
        cmds.append([nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src),
                     "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        for cmd, r in ex.map(run, cmds):
            if verbose or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    tmp = LIB + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        print(r.stdout + r.stderr)
        raise RuntimeError("link of libcp_attn.so failed")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
