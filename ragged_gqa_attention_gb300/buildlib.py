"""Build the CUDA library (librga.so) in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel and the
objects are linked into ``ragged_gqa_attention_gb300/lib/librga.so``.  A
rebuild happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "librga.so")
# The debug-checks variant: every kernel checks its TMA coordinates and
# direct global accesses against their tensors (RGA_DEBUG_CHECKS); a
# violation sets device status 7 and skips the access.
DEBUG_OBJ_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "librga_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(path=None) -> bool:
    path = path or LIB_PATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src, extra, obj_dir=None):
    obj = os.path.join(obj_dir or OBJ_DIR, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, extra_flags=(), jobs=None, debug_checks: bool = False) -> str:
    """Compile and link librga.so (librga_debug.so with debug_checks);
    returns its path."""
    lib_path = DEBUG_LIB_PATH if debug_checks else LIB_PATH
    obj_dir = DEBUG_OBJ_DIR if debug_checks else OBJ_DIR
    if debug_checks:
        extra_flags = tuple(extra_flags) + ("-DRGA_DEBUG_CHECKS",)
    if not force and (debug_checks or not extra_flags) and up_to_date(lib_path):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags), obj_dir), srcs))
    tmp = lib_path + f".{os.getpid()}.tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force=True, debug_checks="--debug-checks" in sys.argv))
