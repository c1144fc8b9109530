"""Builds libwise.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ compiles in parallel; the objects are linked
into block_sparse_paged_split_gb300/lib/libwise.so.  A stamp of the sources,
headers and flags skips the build when nothing changed.  Run as
`python -m block_sparse_paged_split_gb300.build [--force]`.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIBRARY = os.path.join(LIBDIR, "libwise.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=default",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwise.so")


def _sources():
    cus = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    hdrs = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return cus, hdrs


def _stamp(cus, hdrs, extra) -> str:
    h = hashlib.sha256()
    for d, names in ((CSRC, cus + hdrs), (INCLUDE, sorted(os.listdir(INCLUDE)))):
        for n in names:
            h.update(n.encode())
            with open(os.path.join(d, n), "rb") as f:
                h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    extra = list(extra_flags or [])
    cus, hdrs = _sources()
    stamp = _stamp(cus, hdrs, extra)
    stamp_file = os.path.join(LIBDIR, "build.stamp")
    if not force and os.path.exists(LIBRARY) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return LIBRARY
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(name):
        obj = os.path.join(objdir, name[:-3] + ".o")
        cmd = [cc] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, name), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(cus), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, cus))
    tmp = LIBRARY + ".tmp"
    res = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIBRARY


if __name__ == "__main__":
    args = sys.argv[1:]
    path = build_library(force="--force" in args, verbose="-v" in args,
                         extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in args else None)
    print(path)
