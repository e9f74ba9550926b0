"""Builds libftmoe.so in this package directory with nvcc for sm_103a.

Usage: python -m quantized_expert_ffn_layer_b300.build [-j N] [--force] [--checks]
Objects go to ./_build (ignored by git); the shared library is placed next to
this file so that it travels with the source tree.  With --checks the same sources
are built with FTMOE_CHECKS=1 into libftmoe_checks.so (objects in ./_build_checks):
the FFN kernels then bound-check every index they read from offsets / sorted_pair /
inv_pos and report a bad one in the device status word instead of using it.
"""
from __future__ import annotations

import argparse
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libftmoe.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++20", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", CSRC, "-I", INCLUDE]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


LIB_CHECKS = os.path.join(PKG, "libftmoe_checks.so")


def build(jobs: int = 8, force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    build_dir = BUILD + ("_checks" if checks else "")
    lib = LIB_CHECKS if checks else LIB
    extra = ["-DFTMOE_CHECKS=1"] if checks else []
    os.makedirs(build_dir, exist_ok=True)
    hs = headers()
    objs = []
    todo = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hs):
            todo.append((src, obj))

    def compile_one(so):
        src, obj = so
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with ThreadPoolExecutor(max_workers=max(1, jobs)) as ex:
        for src, r in ex.map(compile_one, todo):
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
            if verbose and (r.stdout or r.stderr):
                sys.stderr.write(r.stdout + r.stderr)
    if force or todo or _stale(lib, objs):
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("-j", type=int, default=os.cpu_count() or 8)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", action="store_true", help="pass -Xptxas -v (registers / spills)")
    ap.add_argument("--checks", action="store_true", help="build libftmoe_checks.so (FTMOE_CHECKS=1)")
    a = ap.parse_args()
    print(build(a.j, a.force, a.v, a.checks))
