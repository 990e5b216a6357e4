"""Build the CUDA library in-tree: nvcc for sm_103a only, no cmake.

    python -m block_scaled_mxfp4_gb300.build [--force] [--verbose-ptxas]

Each .cu under csrc/ compiles to an object in parallel, then one link makes
libmxfp4_gb300.so next to this file.  The benchmark's streaming-read helper
(probe/stream_read.cu, not part of the library) links into libmxfp4_probe.so.
Rebuilds only when a source or header is newer than its library.
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmxfp4_gb300.so")
PROBE_SRC = os.path.join(PKG, "probe", "stream_read.cu")
PROBE_LIB = os.path.join(PKG, "libmxfp4_probe.so")
OBJDIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I" + INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + \
        [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build_probe(force: bool = False) -> str:
    """The benchmark's streaming-read helper library."""
    if not force and os.path.exists(PROBE_LIB) and \
            os.path.getmtime(PROBE_SRC) <= os.path.getmtime(PROBE_LIB):
        return PROBE_LIB
    tmp = PROBE_LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-shared", "-o", tmp, PROBE_SRC, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed on the stream-read helper")
    os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not verbose_ptxas and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    # One builder at a time (parallel test workers share the object files);
    # a process that waited finds the library fresh and returns.
    with open(os.path.join(OBJDIR, "build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and not verbose_ptxas and up_to_date():
            return LIB
        return _build_locked(verbose_ptxas)


def _build_locked(verbose_ptxas: bool) -> str:
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src):
        obj = os.path.join(OBJDIR, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    objs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        for src, obj, r in ex.map(compile_one, _sources()):
            if r.returncode != 0 or verbose_ptxas:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
            objs.append(obj)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv))
    print(build_probe(force="--force" in sys.argv))
