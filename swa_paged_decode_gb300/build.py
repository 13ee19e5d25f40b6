"""Build libdsa_decode.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel to an object under
``_build/``; the objects link into ``lib/libdsa_decode.so`` (CUDA runtime
linked statically, so the library only needs the driver). Run as
``python -m swa_paged_decode_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libdsa_decode.so")
# The checking build (-DDSA_DEBUG): every global and tile access bounds-checked.
LIB_DEBUG = os.path.join(LIBDIR, "libdsa_decode_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa_decode.so")
    return p


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(lib: str, deps) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Build the release library, or with ``debug`` the checking build."""
    srcs = sources()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "dsa_decode.h"))
    lib = LIB_DEBUG if debug else LIB
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    if not force and not extra_flags and not _stale(lib, srcs + headers + [__file__]):
        return lib
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if debug:
        flags.append("-DDSA_DEBUG")
    procs = []
    for s in srcs:
        obj = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        log = open(obj + ".log", "w")
        procs.append((s, obj, log, subprocess.Popen([nvcc(), *flags, "-c", s, "-o", obj],
                                                    stdout=log, stderr=subprocess.STDOUT)))
    failed = []
    for s, obj, log, pr in procs:
        pr.wait()
        log.close()
        if pr.returncode != 0:
            failed.append(s)
        if verbose or pr.returncode != 0:
            with open(obj + ".log") as f:
                sys.stderr.write(f.read())
    if failed:
        raise RuntimeError(f"nvcc failed for: {', '.join(os.path.basename(f) for f in failed)}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *[p[1] for p in procs]], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
