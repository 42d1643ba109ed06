"""Build libsparsp.so in-tree for sm_103a with nvcc (no CMake).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
block_sparse_attention_token_gb300/libsparsp.so with the CUDA runtime linked
statically, so loading the library needs no CUDA driver (the ABI checks run
on machines without a GPU).

build(debug=True) makes libsparsp_debug.so instead, compiled with
-DSPARSP_DEBUG: its kernels also check every address they derive themselves
(TMA coordinates, output rows, list and CSR write positions) and report
SPARSP_ERR_DATA rather than use one out of range. The binding loads it when
the environment sets SPARSP_DEBUG=1.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsparsp.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libsparsp_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".h", ".cuh")):
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _compile(src: str, extra: list[str], verbose: bool, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr}")
    if verbose and res.stderr:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    """Compile every CUDA source and link libsparsp.so (libsparsp_debug.so with
    debug=True); returns its path."""
    extra = list(extra or []) + (["-DSPARSP_DEBUG"] if debug else [])
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    stamp_path = os.path.join(build_dir, "stamp")
    srcs = _sources()
    key = hashlib.sha256()
    for s in srcs:
        with open(s, "rb") as fh:
            key.update(s.encode() + fh.read())
    key.update(_headers_digest().encode() + " ".join(ARCH + NVCC_FLAGS + extra).encode())
    stamp = key.hexdigest()
    if not force and os.path.exists(lib) and os.path.exists(stamp_path):
        with open(stamp_path) as fh:
            if fh.read() == stamp:
                return lib
    workers = min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose, build_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as fh:
        fh.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
