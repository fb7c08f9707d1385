"""Build step of the CUDA library ``_lib/libzero.so`` (sm_103a only).

Each translation unit compiles in parallel with nvcc (``-gencode
arch=compute_103a,code=sm_103a -lineinfo -O3 --fmad=false``: no multiply-add
contraction, IEEE division and square root, no fast-math), then nvcc links a
shared library with the CUDA runtime linked statically.  The library is built
in-tree, next to the Python binding that loads it.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_lib", "obj")
LIB = os.path.join(PKG, "_lib", "libzero.so")

CUDA_SOURCES = ["fused_step.cu", "gather.cu", "gen.cu", "clip.cu", "noalloc.cu", "reshard.cu"]
HOST_SOURCES = ["host.cpp", "zero3_sched.cpp", "graph.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
CUDA_FLAGS = ARCH + ["-lineinfo", "--fmad=false", "-Xptxas", "-v"] + COMMON


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero.so")
    return exe


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "zero.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def _compile(src, log):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    flags = CUDA_FLAGS if src.endswith(".cu") else COMMON
    cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append("$ " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr))
    return obj


def build(force=False, verbose=False):
    """Compile and link libzero.so if it is missing or older than its sources."""
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    log = []
    with cf.ThreadPoolExecutor(max_workers=len(CUDA_SOURCES) + len(HOST_SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, log), CUDA_SOURCES + HOST_SOURCES))
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    log.append("$ " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stderr)
    os.replace(tmp, LIB)
    with open(os.path.join(PKG, "_lib", "build.log"), "w") as f:
        f.write("\n".join(log))
    if verbose:
        print("\n".join(log))
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
