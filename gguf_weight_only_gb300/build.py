"""Build the CUDA library (libqlinear.so) in-tree with nvcc for sm_103a only.

Each .cu file under csrc/ compiles to an object in parallel; the objects link into
gguf_weight_only_gb300/_lib/libqlinear.so with the static CUDA runtime. No cmake, no
torch extension machinery: the library exposes the plain C ABI of include/qlinear.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB = os.path.join(OUT_DIR, "libqlinear.so")
# The QL_DEBUG build: every kernel checks the shared- and global-memory ranges its pipelines
# touch, records a failed check in the device status word (QL_ERR_BOUNDS) and skips the access.
DEBUG_OUT_DIR = os.path.join(HERE, "_lib_debug")
DEBUG_LIB = os.path.join(DEBUG_OUT_DIR, "libqlinear.so")


def lib_path(debug: bool = False) -> str:
    return DEBUG_LIB if debug else LIB
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *extra]


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a and link libqlinear.so; returns the library path.
    debug=True builds the bounds-checking QL_DEBUG library into _lib_debug/ instead."""
    deps = _deps() + [os.path.abspath(__file__)]
    lib, obj_dir = (DEBUG_LIB, os.path.join(DEBUG_OUT_DIR, "obj")) if debug else (LIB, OBJ_DIR)
    if debug:
        extra_flags = (*extra_flags, "-DQL_DEBUG")
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *_flags(extra_flags), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
