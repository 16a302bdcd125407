"""Builds libhq.so (the CUDA kernels and their C ABI) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel to an object under ``_build/``
and linked into ``libhq.so`` next to this file.  A stamp of the sources, the
flags and the machine architecture decides whether a rebuild is needed, so a
library compiled on another machine is never reused.

``build(debug=True)`` makes ``libhq_debug.so`` from the same sources with
``-DHQ_DEBUG=1``: the kernels then check the data-dependent indices of their
global writes, set HQ_STATUS_BOUNDS in the device status word when one is
out of range and skip that access (objects under ``_build/debug/``).
"""

import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libhq.so")
STAMP = os.path.join(BUILD_DIR, "libhq.stamp")
DEBUG_BUILD_DIR = os.path.join(BUILD_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(HERE, "libhq_debug.so")
DEBUG_STAMP = os.path.join(DEBUG_BUILD_DIR, "libhq_debug.stamp")

SOURCES = ["hq_common.cu", "hq_quant.cu", "hq_gemm_bs.cu", "hq_gemm_dswiglu.cu", "hq_permute.cu"]
HEADERS = ["hq_ptx.cuh", "hq_internal.h", "hq_sched.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr"]


def nvcc_path():
    p = shutil.which("nvcc")
    if p:
        return p
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhq.so")


def _flags(debug):
    return ARCH + CFLAGS + (["-DHQ_DEBUG=1"] if debug else [])


def _paths(debug):
    return (DEBUG_BUILD_DIR, DEBUG_LIB_PATH, DEBUG_STAMP) if debug else (BUILD_DIR, LIB_PATH, STAMP)


def _stamp(debug=False):
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(_flags(debug)).encode())
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    with open(os.path.join(INCLUDE, "hq.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def up_to_date(debug=False):
    _, lib, stamp = _paths(debug)
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == _stamp(debug)


def build(force=False, verbose=False, debug=False):
    """Compile and link libhq.so (libhq_debug.so with debug=True) if needed;
    returns its path."""
    build_dir, lib_path, stamp = _paths(debug)
    if not force and up_to_date(debug):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = nvcc_path()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc] + _flags(debug) + ["-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
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
        msg = "\n".join(f"--- {s} ---\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib_path + ".tmp"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(_stamp(debug))
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
