"""Build libmk.so in-tree: nvcc for the CUDA translation units (sm_103a only),
g++ for the host planner, compiled in parallel, linked with nvcc -shared
(static CUDA runtime).  Objects go to ``_build/``; the library lands next to
this file.  Rebuilds only when a source or header is newer than the library.

The same build also makes libmk_bounds.so: the C ABI and the small-model
kernel variant (hidden 256) compiled with MK_BOUNDS defined, so that every
checked access of the kernel records MK_ERR_BOUNDS instead of leaving its
buffer (a stand-in for a memory checker; see mk_device.cuh).  The binding
loads it instead of libmk.so when the environment sets MK_LIB=bounds.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmk.so")
LIB_BOUNDS = os.path.join(PKG, "libmk_bounds.so")
# translation units of the bounds-checked library (the small variant only)
BOUNDS_CU = ("api.cu", "pack.cu", "k_h256_d64_g2_b1.cu")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "-Xptxas", "-v"]
CXX_FLAGS = ["-std=c++17", "-O2", "-fPIC", "-Wall", "-I", INCLUDE]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmk.so")
    return p


def _sources():
    cu = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    cpp = sorted(glob.glob(os.path.join(CSRC, "*.cpp")))
    return cu, cpp


def _deps():
    return glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    for lib in (LIB, LIB_BOUNDS):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if not all(os.path.getmtime(f) <= t for f in _deps()):
            return False
    return True


def _compile(cmd, log_path):
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log_path, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp = _sources()
    tasks = []
    objs = []
    for src in cu:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        tasks.append(([nvcc] + NVCC_FLAGS + ["-c", src, "-o", obj], obj + ".log"))
    for src in cpp:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        tasks.append((["g++"] + CXX_FLAGS + ["-c", src, "-o", obj], obj + ".log"))
    bdir = os.path.join(BUILD, "bounds")
    os.makedirs(bdir, exist_ok=True)
    bobjs = [os.path.join(BUILD, os.path.basename(src) + ".o") for src in cpp]  # planner: shared
    for name in BOUNDS_CU:
        src = os.path.join(CSRC, name)
        obj = os.path.join(bdir, name + ".o")
        bobjs.append(obj)
        tasks.append(([nvcc] + NVCC_FLAGS + ["-DMK_BOUNDS=1", "-c", src, "-o", obj], obj + ".log"))
    jobs = jobs or min(len(tasks), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        outs = list(ex.map(lambda t: _compile(*t), tasks))
    if verbose:
        for o in outs:
            for line in o.splitlines():
                if "registers" in line or "spill" in line:
                    print(line)
    for lib, ob in ((LIB, objs), (LIB_BOUNDS, bobjs)):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + ob, check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
