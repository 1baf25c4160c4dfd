"""Builds the layer's CUDA library (libmoe_gb300.so) in-tree for sm_103a.

Every .cu file under csrc/ is compiled by nvcc in parallel, then linked into
one shared library exporting the C ABI of include/moe.h.  Rebuilds only when a
source or header is newer than the library.
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libmoe_gb300.so")
# the bounds-checked debug build (-DMOE_DEBUG): same sources and ABI
OUT_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(OUT_DEBUG, "libmoe_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force=False, verbose=False, extra=(), debug=False):
    """Compile and link; returns the library path.  Raises on compiler errors.
    debug=True builds the bounds-checked variant (-DMOE_DEBUG) into its own
    directory."""
    out, lib = (OUT_DEBUG, LIB_DEBUG) if debug else (OUT, LIB)
    extra = tuple(extra) + (("-DMOE_DEBUG",) if debug else ())
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src).replace(".cu", ".o"))
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
