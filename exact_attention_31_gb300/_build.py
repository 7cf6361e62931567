"""Build libfattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

The translation units are compiled in parallel and linked into one shared library that
exports the C ABI declared in include/fattn.h.  The same sources built with -DFATTN_DEBUG give
libfattn_debug.so, whose kernels check every TMA, tensor-memory and barrier operand and every output
store before they issue it (fattn.h, "Debug builds"); both are built together.  The standard
three-kernel attention that the fused forward is measured against (fattn_unfused.h) is a library of
its own, libfattn_unfused.so, linked against cuBLAS; libfattn does not depend on it.
"""

from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfattn.so")
STAMP = os.path.join(BUILD, "libfattn.stamp")
DEBUG_BUILD = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libfattn_debug.so")
DEBUG_STAMP = os.path.join(DEBUG_BUILD, "libfattn_debug.stamp")
DEBUG_FLAGS = ["-DFATTN_DEBUG"]
UNFUSED_BUILD = os.path.join(PKG, "_build_unfused")
UNFUSED_LIB = os.path.join(PKG, "libfattn_unfused.so")
UNFUSED_STAMP = os.path.join(UNFUSED_BUILD, "libfattn_unfused.stamp")

SOURCES = ["fattn_api.cu", "prefill_sm103a.cu", "prefill_fp8_sm103a.cu", "decode_sm103a.cu", "backward_sm103a.cu",
           "host_staging.cu", "mask_tiles_sm103a.cu"]
HEADERS = ["fattn_internal.h", "sm103a_ptx.cuh"]
UNFUSED_SOURCES = ["unfused_sm103a.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--use_fast_math", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cuda_lib_dir() -> str:
    """The CUDA toolkit's library directory, next to the nvcc in use (cuBLAS for the unfused library)."""
    return os.path.realpath(os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64"))


def _sources(unfused: bool):
    return UNFUSED_SOURCES if unfused else SOURCES


def _link_flags(unfused: bool):
    if not unfused:
        return []
    d = cuda_lib_dir()
    return ["-L", d, "-lcublas", "-Xlinker", f"-rpath,{d}"]


def _inputs(unfused: bool = False):
    files = [os.path.join(CSRC, s) for s in _sources(unfused) + ([] if unfused else HEADERS)]
    files.append(os.path.join(INCLUDE, "fattn.h"))
    if unfused:
        files.append(os.path.join(INCLUDE, "fattn_unfused.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_digest(extra_flags=None, unfused: bool = False) -> str:
    """Hash of everything the library is built from: the sources, the headers, this file, the flags,
    the compiler's path and the host architecture (a library built on another machine never
    matches)."""
    h = hashlib.sha256()
    for f in _inputs(unfused):
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags or []) + _link_flags(unfused)).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _paths(debug: bool, unfused: bool = False):
    if unfused:
        return UNFUSED_BUILD, UNFUSED_LIB, UNFUSED_STAMP
    return (DEBUG_BUILD, DEBUG_LIB, DEBUG_STAMP) if debug else (BUILD, LIB, STAMP)


def _flags(debug: bool, extra_flags=None):
    return (DEBUG_FLAGS if debug else []) + list(extra_flags or [])


def up_to_date(extra_flags=None, debug: bool = False, unfused: bool = False) -> bool:
    """True when the library exists and was built here from exactly the current sources."""
    _, lib, stamp = _paths(debug, unfused)
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        return f.read().strip() == source_digest(_flags(debug, extra_flags), unfused)


def _start(debug: bool, extra_flags, verbose: bool, unfused: bool = False):
    """Start the nvcc processes of one variant; returns what _finish needs."""
    build_dir, _, _ = _paths(debug, unfused)
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + _flags(debug, extra_flags)
    procs = []
    objs = []
    for src in _sources(unfused):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    return debug, extra_flags, procs, objs, unfused


def _finish(job, verbose: bool) -> str:
    debug, extra_flags, procs, objs, unfused = job
    _, lib, stamp = _paths(debug, unfused)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}" + (" (debug build)" if debug else ""))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, *_link_flags(unfused)], check=True)
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(source_digest(_flags(debug, extra_flags), unfused) + "\n")
    return lib


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug: bool = False) -> str:
    """Build one variant (the release library, or with debug=True the checked one)."""
    if not force and up_to_date(extra_flags, debug):
        return _paths(debug)[1]
    return _finish(_start(debug, extra_flags, verbose), verbose)


def build_unfused(force: bool = False, verbose: bool = False) -> str:
    """Build libfattn_unfused.so (the standard three-kernel attention)."""
    if not force and up_to_date(unfused=True):
        return UNFUSED_LIB
    return _finish(_start(False, None, verbose, unfused=True), verbose)


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Build the release, debug and unfused libraries, all translation units compiled at once."""
    jobs = [_start(d, None, verbose) for d in (False, True) if force or not up_to_date(None, d)]
    if force or not up_to_date(unfused=True):
        jobs.append(_start(False, None, verbose, unfused=True))
    for job in jobs:
        _finish(job, verbose)


if __name__ == "__main__":
    build_all(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
    print(DEBUG_LIB)
    print(UNFUSED_LIB)
