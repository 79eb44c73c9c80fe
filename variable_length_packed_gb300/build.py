"""Build libthdattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically, so the library loads on a
machine without a GPU driver (its calls then return THD_ERR_CUDA) and has no
link-time dependency on libcuda (the TMA encoder is fetched through the
runtime's driver entry-point query).
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libthdattn.so")
BUILD_DIR = os.path.join(PKG, "_build")
# content hash of the sources and flags the library was built from, written beside it
STAMP = LIB + ".sha256"

SOURCES = ["thd_attn.cu", "padding_mask.cu", "attn_noalloc.cu", "attn_merge.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libthdattn.so")
    return exe


def source_hash(extra_flags=()):
    """SHA-256 over every file under csrc/ and include/ (names and contents, sorted) and the
    compiler flags: the library is rebuilt whenever any of them differs from what it was
    built from, whatever the files' times say."""
    h = hashlib.sha256()
    for d in (CSRC, os.path.join(ROOT, "include")):
        for f in sorted(os.listdir(d)):
            path = os.path.join(d, f)
            if os.path.isfile(path):
                h.update(os.path.relpath(path, ROOT).encode() + b"\0")
                with open(path, "rb") as fh:
                    h.update(fh.read())
                h.update(b"\0")
    h.update(" ".join([*ARCH, *FLAGS, *extra_flags]).encode())
    return h.hexdigest()


def _stale(extra_flags=()):
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        return f.read().strip() != source_hash(extra_flags)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile (if needed) and return the path of libthdattn.so."""
    extra = list(extra_flags or [])
    if not force and not _stale(extra):
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    digest = source_hash(extra)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stdout.write(out)
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest + "\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)
