"""Builds libssm.so in-tree with nvcc for sm_103a (B300)."""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libssm.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]
OBJ_DIR = os.path.join(PKG_DIR, "_build")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ (one nvcc process per file, in parallel) and link them
    into libssm.so if any source is newer than it."""
    stale = force or not os.path.exists(LIB_PATH) or any(
        os.path.getmtime(LIB_PATH) < os.path.getmtime(s) for s in _deps())
    if stale:
        os.makedirs(OBJ_DIR, exist_ok=True)
        objs = [os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o") for src in sources()]

        def compile_one(src, obj):
            cmd = [NVCC, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj, src]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            subprocess.run(cmd, check=True)

        with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
            for f in [ex.submit(compile_one, s, o) for s, o in zip(sources(), objs)]:
                f.result()
        subprocess.run([NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o",
                        LIB_PATH + ".tmp", *objs], check=True)
        os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH
