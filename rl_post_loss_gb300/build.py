"""Builds ``librl_loss.so`` from ``csrc/`` with nvcc for sm_103a.

Each translation unit compiles in parallel, then one nvcc call links the
shared library (static CUDA runtime, only the ``rl_loss_*`` symbols exported).
The library is written next to this file (in-tree) and is git-ignored.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "librl_loss.so")
# The debug build: every kernel also checks its index invariants and raises RL_ERR_INTERNAL
# (skipping the access) where one fails. Built on request, next to the normal library.
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(HERE, "librl_loss_debug.so")
DEBUG_FLAGS = ["-DRL_LOSS_DEBUG_CHECKS"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def nvcc_path() -> str:
    import shutil
    n = nvcc()
    return n if os.path.isabs(n) else (shutil.which(n) or "/usr/local/cuda/bin/nvcc")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None, debug: bool = False) -> str:
    build_dir, lib_path = (DEBUG_BUILD_DIR, DEBUG_LIB_PATH) if debug else (BUILD_DIR, LIB_PATH)
    if debug:
        extra_flags = DEBUG_FLAGS + (extra_flags or [])
    os.makedirs(build_dir, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    srcs = sources()
    objs = []
    procs = []
    flags = NVCC_FLAGS + (extra_flags or [])
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc()] + ARCH + flags + ["-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"--- {s}\n{o}" for s, o in failed))
    if force or procs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        subprocess.check_call(cmd)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
