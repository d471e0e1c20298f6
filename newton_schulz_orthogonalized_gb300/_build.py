"""Builds libnsmuon.so in-tree with nvcc for sm_103a (no torch extension machinery).

Each translation unit compiles in its own nvcc process (in parallel), then one link
step makes the shared library next to this file.  The checked build,
libnsmuon_checked.so, is the same sources compiled with NSM_CHECKED=1: its kernels test
every access to a matrix's elements (global loads and stores, TMA boxes) against that
matrix before making it, record a failure in the device status word and skip the access.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libnsmuon.so")
LIB_CHECKED = os.path.join(HERE, "libnsmuon_checked.so")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
SOURCES = ["nsm_api.cpp", "elementwise.cu", "ns_gemm.cu", "ns_small.cu", "status_check.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def _jobs(checked: bool, ptxas_info: bool):
    """(compile commands, objects, link command pieces, output) of one library."""
    nvcc = _nvcc()
    out_dir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(out_dir, exist_ok=True)
    defs = ["-DNSM_CHECKED=1"] if checked else []
    objs, cmds = [], []
    for src in SOURCES:
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc] + ARCH + COMMON + defs + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd += ["-x", "cu"]
        if ptxas_info and src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        cmds.append(cmd)
    return cmds, objs, LIB_CHECKED if checked else LIB


def _link(objs, lib):
    tmp = lib + ".tmp"
    _run([_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, lib)


def build(verbose: bool = False, ptxas_info: bool = False, checked: bool = False,
          both: bool = False) -> str:
    """Builds libnsmuon.so (or, with checked, libnsmuon_checked.so; with both, the two
    at once, their translation units compiled in parallel).  Returns the regular
    library's path (the checked one's when only it is built)."""
    variants = [False, True] if both else [checked]
    jobs = [_jobs(c, ptxas_info) for c in variants]
    cmds = [c for j in jobs for c in j[0]]
    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for o in outs:
            if o.strip():
                print(o)
    for _, objs, lib in jobs:
        _link(objs, lib)
    return jobs[0][2]


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, checked="--checked" in sys.argv,
                both="--both" in sys.argv))
