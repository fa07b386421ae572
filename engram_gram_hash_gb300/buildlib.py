"""Builds libengram.so in-tree with nvcc for sm_103a (one translation unit)."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC_DIR = os.path.join(HERE, "csrc")
MAIN_SRC = os.path.join(SRC_DIR, "engram_core.cu")
LIB_PATH = os.path.join(HERE, "libengram.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    out = []
    for d in (SRC_DIR, os.path.join(os.path.dirname(HERE), "include")):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                out.append(os.path.join(d, f))
    return out


def build_cmd(out=LIB_PATH, extra=()):
    return [
        "nvcc", *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
        *extra, "-o", out, MAIN_SRC,
    ]


def build(force=False, verbose=False):
    """Compile if any source is newer than the library; returns its path."""
    stale = force or not os.path.exists(LIB_PATH)
    if not stale:
        t = os.path.getmtime(LIB_PATH)
        stale = any(os.path.getmtime(s) > t for s in sources())
    if stale:
        cmd = build_cmd()
        if verbose:
            print(" ".join(cmd))
        subprocess.check_call(cmd)
    return LIB_PATH
