"""Compile libmoe.so from csrc/*.cu with nvcc for sm_103a (in-tree build).

Each translation unit compiles to an object in parallel; the objects link
into one shared library next to this file. No torch C++ headers are used, so
the library loads with plain ctypes.

An object is rebuilt unless its stamp file records the same key: a hash of
nvcc's version banner, the architecture and flags, and the contents of the
source and of every header it may include. So a changed flag, another nvcc or
an object copied in from elsewhere never reuses stale code, whatever the files'
modification times say.
"""
from __future__ import annotations

import concurrent.futures as cf
import functools
import glob
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libmoe.so")
BUILD_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dirs(nvcc: str):
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    dirs = [os.path.join(root, "lib64"), os.path.join(root, "targets", "sbsa-linux", "lib"),
            os.path.join(root, "targets", "x86_64-linux", "lib")]
    dirs += [os.path.join(d, "stubs") for d in list(dirs)]
    return [d for d in dirs if os.path.isdir(d)]


@functools.lru_cache(maxsize=None)
def _nvcc_banner(nvcc: str) -> str:
    return subprocess.run([nvcc, "--version"], capture_output=True, text=True,
                          check=True).stdout


def _key(nvcc: str, cmd, src: str, deps) -> str:
    h = hashlib.sha256()
    h.update(_nvcc_banner(nvcc).encode())
    h.update("\0".join(cmd).encode())
    for p in [src, *deps]:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(hashlib.sha256(f.read()).digest())
    return h.hexdigest()


def _stale(obj: str, key: str) -> bool:
    stamp = obj + ".key"
    if not (os.path.exists(obj) and os.path.exists(stamp)):
        return True
    with open(stamp) as f:
        return f.read().strip() != key


def build(verbose: bool = False, force: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "moe.h")]
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        flags = [*ARCH, *NVFLAGS, "-c", os.path.basename(src)]
        key = _key(nvcc, flags, src, deps)
        if force or _stale(obj, key):
            jobs.append(([nvcc, *ARCH, *NVFLAGS, "-c", src, "-o", obj], obj, key))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("nvcc failed: " + " ".join(cmd))

    def compile_one(job):
        cmd, obj, key = job
        stamp = obj + ".key"
        if os.path.exists(stamp):
            os.remove(stamp)
        run(cmd)
        with open(stamp, "w") as f:
            f.write(key + "\n")

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(compile_one, jobs))
    objs = [os.path.join(BUILD_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    # The library's key: every object's key and the link flags.
    h = hashlib.sha256(" ".join([*ARCH, "-shared", "-cudart", "static"]).encode())
    for o in objs:
        with open(o + ".key") as f:
            h.update(f.read().encode())
    lib_key = h.hexdigest()
    lib_stamp = os.path.join(BUILD_DIR, "libmoe.so.key")
    if force or jobs or _stale_lib(lib_stamp, lib_key):
        libdirs = [f"-L{d}" for d in _cuda_lib_dirs(nvcc)]
        tmp = LIB + f".{os.getpid()}.tmp"
        if os.path.exists(lib_stamp):
            os.remove(lib_stamp)
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, *libdirs, "-cudart", "static"])
        os.replace(tmp, LIB)
        with open(lib_stamp, "w") as f:
            f.write(lib_key + "\n")
    return LIB


def _stale_lib(stamp: str, key: str) -> bool:
    if not (os.path.exists(LIB) and os.path.exists(stamp)):
        return True
    with open(stamp) as f:
        return f.read().strip() != key


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
