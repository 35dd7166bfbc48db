"""Build libmoe.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m sparse_conditional_moe_b300.build [--force] [--verbose]

Each csrc/*.cu is compiled to an object under _build/, then everything is linked into
sparse_conditional_moe_b300/libmoe.so with the static CUDA runtime.  The library depends on
nothing else at load time (the driver is reached through the runtime), so it also loads on a
machine without a GPU.

Rebuilds are keyed on content, not on file times: every object carries the SHA-256 of the
compiler's version, the flags, its source and every header, and the library carries the hash
of its objects' keys and the link line (`libmoe.so.key` beside it).  A library whose key
matches the sources is up to date even where no object exists (a fresh checkout that received
the built library); any change to a source, a header, a flag or the compiler rebuilds what it
touches.  Objects compile in parallel.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe.so")
LIB_KEY = LIB + ".key"
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]
LINK = ["-shared", "-cudart", "static"]


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _read(path: str) -> bytes:
    with open(path, "rb") as f:
        return f.read()


def _nvcc_version() -> bytes:
    return subprocess.run([NVCC, "--version"], check=True, capture_output=True).stdout


def _object_key(src: str, common: bytes) -> str:
    h = hashlib.sha256(common)
    h.update(os.path.basename(src).encode())
    h.update(_read(src))
    return h.hexdigest()


def _stored(path: str) -> str:
    try:
        with open(path) as f:
            return f.read().strip()
    except OSError:
        return ""


def _write(path: str, text: str) -> None:
    tmp = path + f".tmp{os.getpid()}"
    with open(tmp, "w") as f:
        f.write(text + "\n")
    os.replace(tmp, path)


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    common = hashlib.sha256()
    common.update(_nvcc_version())
    common.update(" ".join(ARCH + FLAGS).encode())
    for hdr in _headers():
        common.update(os.path.relpath(hdr, ROOT).encode())
        common.update(_read(hdr))
    common = common.digest()
    keys = {src: _object_key(src, common) for src in srcs}
    lib_key = hashlib.sha256(("\n".join(keys[s] for s in srcs) + " ".join(ARCH + LINK)).encode()).hexdigest()
    if not force and os.path.exists(LIB) and _stored(LIB_KEY) == lib_key:
        if verbose:
            print(f"libmoe.so up to date (key {lib_key[:16]})", flush=True)
        return LIB

    os.makedirs(BUILD, exist_ok=True)
    objs, todo = [], []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or _stored(obj + ".key") != keys[src]:
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        _write(obj + ".key", keys[src])

    workers = max(1, min(len(todo), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        for f in [ex.submit(compile_one, it) for it in todo]:
            f.result()
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *LINK, "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    _write(LIB_KEY, lib_key)
    if verbose:
        print(f"built libmoe.so ({len(todo)} of {len(srcs)} objects compiled, key {lib_key[:16]})",
              flush=True)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(a.force, a.verbose))
    sys.exit(0)
