"""Builds libnvfp4_gb300.so in-tree with nvcc for sm_103a (GB300).

Each .cu under csrc/ compiles to an object in parallel, then one shared
library is linked.  Nothing is installed; the library lands in
nvfp4_block_scale_gb300/_build/ (git-ignored) and is rebuilt when a source or
header is newer than it.  build(checked=True) makes the bounds-checked variant
(-DNVFP4_CHECKED, libnvfp4_gb300_checked.so, objects under _build/checked/).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libnvfp4_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
# the checked build (-DNVFP4_CHECKED: bounds-checked kernel accesses, for tests)
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "libnvfp4_gb300_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")
    return found


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles and links the library (with checked=True the -DNVFP4_CHECKED
    variant, beside it); returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and up_to_date(lib_path):
        return lib_path
    obj_dir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    os.makedirs(obj_dir, exist_ok=True)
    exe = nvcc()
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(exe)), "lib64")
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe] + NVCC_FLAGS + (["-DNVFP4_CHECKED"] if checked else []) + \
            (["-Xptxas", "-v"] if verbose else []) + ["-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out)
        if p.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [exe] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + \
        ["-Xlinker", "-rpath," + cuda_lib]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
