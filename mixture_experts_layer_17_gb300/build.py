"""Builds libmoe.so in-tree with nvcc for sm_103a.

Each .cu file of csrc/ is compiled to an object in parallel (objects are
reused while they are newer than every source and header), then linked into
``mixture_experts_layer_17_gb300/lib/libmoe.so`` with the CUDA runtime linked
statically.  No cmake, one -gencode.

``build(checked=True)`` builds the debug variant ``lib/libmoe_checked.so``
with -DMOE_DEVICE_CHECKS: the kernels check every index they read from memory
(expert ids, permuted rows, (token, slot) rows) and record an out-of-range one
in the status word instead of using it.  Setting LIBMOE_PATH to it makes the
binding load it instead of libmoe.so.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libmoe.so")
CHECKED_LIB_PATH = os.path.join(LIB_DIR, "libmoe_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "-I", CSRC] + ARCH


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(f) for f in files), default=0.0)


def _compile(src: str, obj: str, verbose: bool, extra=()) -> None:
    cmd = [_nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stderr}")


def build(verbose: bool = False, force: bool = False, checked: bool = False) -> str:
    """Compiles and links libmoe.so (or, checked, libmoe_checked.so); returns its path."""
    build_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    extra = ["-DMOE_DEVICE_CHECKS"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = _deps_mtime()
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or \
                os.path.getmtime(obj) < max(os.path.getmtime(src), deps):
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for f in [ex.submit(_compile, s, o, verbose, extra) for s, o in jobs]:
                f.result()
    newest = max(os.path.getmtime(o) for o in objs)
    if force or jobs or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest:
        cmd = [_nvcc(), "-shared", "-cudart", "static"] + ARCH + objs + ["-o", lib_path]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib_path)} failed:\n{res.stderr}")
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
