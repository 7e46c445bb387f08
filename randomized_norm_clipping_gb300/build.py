"""Builds libdprc.so in-tree from the CUDA sources in csrc/ (sm_103a only),
and its bounds-checked variant libdprc_debug.so (the same sources with
DPRC_DEBUG defined: every computed global or distributed-shared-memory index
is checked before its access, a failed check is recorded in the device error
word and the access skipped).

Every translation unit of both variants is compiled in parallel, then each
variant is linked into one shared library next to this file.  Run
``python -m randomized_norm_clipping_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libdprc.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libdprc_debug.so")

SOURCES = ["api.cu", "tc_proj.cu", "tc_exact.cu", "tc_narrow.cu", "tc_hutch.cu", "simt.cu", "qr.cu", "qr_cluster.cu", "hutchpp.cu", "noise.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
VARIANTS = {"release": ([], LIB_PATH), "debug": (["-DDPRC_DEBUG"], DEBUG_LIB_PATH)}


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags():
    return ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
            "-I" + INCLUDE, "-I" + CSRC]


def _compile(job):
    variant, src = job
    out_dir = os.path.join(BUILD_DIR, variant)
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *_flags(), *VARIANTS[variant][0], "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
    return obj


def _link(objs, path):
    tmp = path + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)


def build(verbose=False, variants=("release", "debug")):
    """Compiles every translation unit of the given variants and links each
    into its shared library; returns the release library's path."""
    for v in variants:
        os.makedirs(os.path.join(BUILD_DIR, v), exist_ok=True)
    jobs = [(v, src) for v in variants for src in SOURCES]
    workers = min(len(jobs), max(4, os.cpu_count() or 4))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(_compile, jobs))
    for v in variants:
        _link([o for (vv, _), o in zip(jobs, objs) if vv == v], VARIANTS[v][1])
        if verbose:
            print("built", VARIANTS[v][1])
    return LIB_PATH


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
