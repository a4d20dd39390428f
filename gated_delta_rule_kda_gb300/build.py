"""Build ``libkda.so`` in-tree with nvcc for sm_103a (GB300).

Each ``csrc/*.cu`` translation unit is compiled in parallel into
``_build/*.o``, then linked into ``_build/libkda.so``.  Objects are rebuilt
only when their source, a shared header or the flags changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libkda.so")
# The debug library: every prefill entry point first runs the contents checks of
# kda_check_prefill_inputs (compiled with KDA_DEBUG defined), built beside the normal one.
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libkda.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _flags(debug: bool) -> list:
    return NVCC_FLAGS + (["-DKDA_DEBUG"] if debug else [])


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda")
    return path


def _headers_digest(debug: bool) -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))):
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(_flags(debug)).encode())
    return h.hexdigest()


def _stamp_path(obj: str) -> str:
    return obj + ".stamp"


def _needs_build(src: str, obj: str, digest: str) -> bool:
    if not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(src):
        return True
    try:
        with open(_stamp_path(obj)) as f:
            return f.read() != digest
    except OSError:
        return True


def _compile(src: str, obj: str, digest: str, debug: bool) -> str:
    cmd = [nvcc(), *_flags(debug), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    with open(_stamp_path(obj), "w") as f:
        f.write(digest)
    with open(obj + ".ptxas.txt", "w") as f:
        f.write(r.stderr)
    return obj


def build(force: bool = False, jobs: int | None = None, verbose: bool = False,
          debug: bool = False) -> str:
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    digest = _headers_digest(debug)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in sources]
    todo = [(s, o) for s, o in zip(sources, objs) if force or _needs_build(s, o, digest)]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda so: _compile(so[0], so[1], digest, debug), todo))
    if todo or not os.path.exists(lib):
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libkda.so failed:\n{r.stderr}")
        os.replace(tmp, lib)
    if verbose:
        for o in objs:
            p = o + ".ptxas.txt"
            if os.path.exists(p):
                print(open(p).read())
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
