"""Build libgdn_b300.so (all CUDA sources under csrc/) in-tree for sm_103a.

Importable without importing the package (it touches nothing but the
compiler), so a clean checkout can be built before the library exists:
    python gated_deltanet_sequence_prefill_b300/build.py [--ptxas-v]
The package's binding calls build() itself when the library is missing or
older than its sources.  Concurrent builders (several ranks importing the
package at once) serialise on a lock file; the library is replaced
atomically, so a reader never sees a half-written file.
"""
import concurrent.futures
import fcntl
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgdn_b300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    return deps + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def stale():
    """True when the library is missing or older than any source it is built from."""
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def _compile(src, objdir, extra, verbose):
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return obj


def build(force=False, verbose=False, extra=()):
    """Compile every csrc/*.cu for sm_103a and link libgdn_b300.so; returns its path."""
    if not force and not stale():
        return LIB
    objdir = os.path.join(PKG, "_build")
    os.makedirs(objdir, exist_ok=True)
    with open(os.path.join(objdir, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        try:
            if not force and not stale():  # another process built it while we waited
                return LIB
            srcs = sources()
            workers = max(1, min(len(srcs), os.cpu_count() or 1))
            with concurrent.futures.ThreadPoolExecutor(workers) as pool:
                objs = list(pool.map(lambda s: _compile(s, objdir, extra, verbose), srcs))
            tmp = LIB + ".tmp%d" % os.getpid()
            subprocess.run([NVCC, *FLAGS, "-shared", "-o", tmp, *objs], check=True)
            os.replace(tmp, LIB)
        finally:
            fcntl.flock(lk, fcntl.LOCK_UN)
    return LIB


if __name__ == "__main__":
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(force=True, verbose=True, extra=extra))
