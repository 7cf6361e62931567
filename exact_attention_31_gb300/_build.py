"""Build libfattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

The translation units are compiled in parallel and linked into one shared library that
exports the C ABI declared in include/fattn.h.
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

SOURCES = ["fattn_api.cu", "prefill_sm103a.cu", "prefill_fp8_sm103a.cu", "decode_sm103a.cu", "backward_sm103a.cu",
           "host_staging.cu", "mask_tiles_sm103a.cu"]
HEADERS = ["fattn_internal.h", "sm103a_ptx.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--use_fast_math", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "fattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_digest(extra_flags=None) -> str:
    """Hash of everything the library is built from: the sources, the headers, this file, the flags,
    the compiler's path and the host architecture (a library built on another machine never
    matches)."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags or [])).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def up_to_date(extra_flags=None) -> bool:
    """True when libfattn.so exists and was built here from exactly the current sources."""
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as f:
        return f.read().strip() == source_digest(extra_flags)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if not force and up_to_date(extra_flags):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(source_digest(extra_flags) + "\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
