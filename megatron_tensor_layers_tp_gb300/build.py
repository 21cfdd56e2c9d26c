"""Builds the in-tree shared library ``_build/libtp_gb300.so`` for sm_103a.

Translation units compile in parallel (one per GEMM epilogue, plus attention,
the small kernels and the host API), then nvcc links them.  No cmake.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libtp_gb300.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
N_EPI = 8


def _units():
    units = []
    for name in ("small", "attention", "tp_api", "no_alloc"):
        units.append((os.path.join(CSRC, name + ".cu"), os.path.join(BUILD, name + ".o"), []))
    for e in range(N_EPI):
        units.append((os.path.join(CSRC, "gemm_inst.cu"), os.path.join(BUILD, f"gemm_epi{e}.o"),
                      [f"-DTPK_EPI={e}"]))
    return units


def _sources_newer(obj: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if os.path.getmtime(os.path.join(d, f)) > t:
                return True
    return False


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    units = _units()
    todo = [u for u in units if force or _sources_newer(u[1])]

    def compile_one(u):
        src, obj, extra = u
        cmd = ["nvcc", *FLAGS, *ARCH, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4) or 1) as ex:
        for cmd, r in ex.map(compile_one, todo):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if todo or not os.path.exists(LIB):
        cmd = ["nvcc", *ARCH, "-shared", "-cudart", "shared", "-o", LIB,
               *[u[1] for u in units]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("link failed")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
