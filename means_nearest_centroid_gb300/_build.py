"""Build libkmassign.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel to an object, then the
objects are linked into one shared library (CUDA runtime linked statically,
no link against libcuda: the driver entry point for TMA descriptors is looked
up at run time).  Outputs go to ``means_nearest_centroid_gb300/_build/``.
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libkmassign.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["api.cu", "assign.cu", "topk.cu", "aux_kernels.cu", "update.cu", "host_path.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkmassign")
    return path


def _deps():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


# The debug build: the same sources with KMASSIGN_DEBUG defined (device-side
# consistency checks that record KMASSIGN_ERR_DEBUG_CHECK), in a library and
# object folder of its own so that it never replaces the normal build.
DEBUG_DIR = os.path.join(BUILD_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(BUILD_DIR, "libkmassign_debug.so")


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile (if stale) and return the path of libkmassign.so (with
    ``debug``: of libkmassign_debug.so, built with KMASSIGN_DEBUG)."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    obj_dir = DEBUG_DIR if debug else BUILD_DIR
    if not force and not extra_flags and up_to_date(lib_path):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags) + (["-DKMASSIGN_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
