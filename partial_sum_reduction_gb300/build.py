"""Builds libshmm.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each translation unit under csrc/ compiles in parallel into _build/, then
they link into partial_sum_reduction_gb300/libshmm.so (CUDA runtime linked
statically, so the library depends only on the driver at run time).

build(checked=True) makes the bounds-checked variant instead: the same
sources compiled with SHMM_CHECKED into _build_checked/ and linked as
libshmm_checked.so, whose kernels compare every global index with its
buffer's extent (a debugging aid; the binding loads it when SHMM_CHECKED=1).
"""
import concurrent.futures
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libshmm.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libshmm_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

SOURCES = ["planner.cpp", "api.cu", "collectives.cu", "gemm_simt.cu", "gemm_tcgen05.cu"]


def _nvcc():
    cand = os.environ.get("NVCC") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers_mtime():
    hs = (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
          glob.glob(os.path.join(INCLUDE, "*.h")))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src, verbose, build_dir, defines):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    path = os.path.join(CSRC, src)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), _headers_mtime()):
        return obj, False
    cmd = [_nvcc()] + ARCH + FLAGS + defines + ["-c", path, "-o", obj + ".tmp"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj, True


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles csrc/*.cu, csrc/*.cpp -> libshmm.so (libshmm_checked.so with
    checked=True); returns the library path."""
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    defines = ["-DSHMM_CHECKED"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for o in glob.glob(os.path.join(build_dir, "*.o")):
            os.remove(o)
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, build_dir, defines), SOURCES))
    objs = [o for o, _ in results]
    changed = any(c for _, c in results)
    if changed or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
