"""Build libfp8kv.so in-tree: every csrc/*.cu compiled for sm_103a with nvcc,
in parallel, then linked into fp8_e4m3_kv_gb300/libfp8kv.so (static cudart).
csrc_probe/*.cu (the benchmark's FP8 tensor-core throughput probe) links
into libfp8kv_probe.so beside it."""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8kv.so")
PROBE_LIB = os.path.join(PKG, "libfp8kv_probe.so")
CSRC_PROBE = os.path.join(PKG, "csrc_probe")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I" + os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _probe_sources():
    return sorted(glob.glob(os.path.join(CSRC_PROBE, "*.cu")))


def _deps():
    return _sources() + _probe_sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(ROOT, "include", "fp8kv.h"), os.path.abspath(__file__)]


def needs_build() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(PROBE_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(PROBE_LIB))
    return any(os.path.getmtime(d) > t for d in _deps())


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC] + ARCH + FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    probe_srcs = _probe_sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs) + len(probe_srcs))) as ex:
        objs = list(ex.map(_compile, srcs + probe_srcs))
    for lib, lib_objs in ((LIB, objs[:len(srcs)]), (PROBE_LIB, objs[len(srcs):])):
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + lib_objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)
    if verbose:
        print("built", LIB, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
