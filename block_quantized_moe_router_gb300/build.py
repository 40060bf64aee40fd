"""Build the CUDA library libmoe_gb300.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and linked with the static CUDA
runtime, so the shared object loads without a GPU (the driver is resolved on first use).

A stamp file beside the library holds a hash of every source, the header, this script, the
compiler flags, the nvcc version and the machine; the library is rebuilt whenever the stamp
does not match (a copied-in library built elsewhere is never reused), and each call says on
stderr whether it compiled or reused the library.
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
SOURCES = ["api.cu", "route.cu", "ffn.cu", "decode.cu", "decode_t1.cu", "prefill_tc.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


STAMP = LIB + ".stamp"
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I",
                CSRC, "--expt-relaxed-constexpr"]


def _nvcc_version() -> str:
    try:
        return subprocess.run([nvcc(), "--version"], capture_output=True, text=True).stdout
    except OSError:
        return "no nvcc"


def source_stamp() -> str:
    """Hash of everything the library is built from, and of where it is built."""
    h = hashlib.sha256()
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    files += [os.path.join(INCLUDE, "moe.h"), os.path.abspath(__file__)]
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(FLAGS).encode())
    h.update(_nvcc_version().encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    stamp = source_stamp()
    if not force and os.path.exists(LIB) and os.path.exists(STAMP):
        with open(STAMP) as fh:
            if fh.read().strip() == stamp:
                sys.stderr.write(f"libmoe_gb300: reused {LIB} (stamp {stamp[:16]})\n")
                return LIB
    flags = list(FLAGS)
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose:
            sys.stderr.write(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as fh:
        fh.write(stamp + "\n")
    sys.stderr.write(f"libmoe_gb300: compiled {LIB} (stamp {stamp[:16]})\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
