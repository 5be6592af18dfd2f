"""Builds the C-ABI shared library ``libattn_bwd.so`` in-tree with nvcc.

Each translation unit under ``csrc/`` is compiled for sm_103a in parallel and
linked with the static CUDA runtime.  A stamp of the sources and flags makes
repeated calls cheap; a missing library, a changed source or a library built
for another machine architecture triggers a rebuild.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn_bwd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC", "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn_bwd.so")
    return path


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            p = os.path.join(d, f)
            if os.path.isfile(p):
                h.update(f.encode())
                with open(p, "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()


# Named builds besides the release library: "debug" compiles every kernel with
# -DATTN_DEBUG (device-side index checks that record a failing check in the
# workspace header and skip the access).
VARIANTS = {"": (), "debug": ("-DATTN_DEBUG",)}


def library_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(PKG, f"libattn_bwd_{variant}.so")


def build_library(verbose: bool = False, extra_flags=(), force: bool = False, variant: str = "") -> str:
    """Compile (if needed) and return the path of libattn_bwd.so (or of a named
    variant, e.g. "debug")."""
    extra_flags = tuple(VARIANTS[variant]) + tuple(extra_flags)
    lib_path = library_path(variant)
    out_dir = OUT_DIR if not variant else os.path.join(OUT_DIR, variant)
    stamp = os.path.join(out_dir, "stamp.txt")
    os.makedirs(out_dir, exist_ok=True)
    digest = _digest(extra_flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib_path
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc] + NVCC_FLAGS + list(extra_flags) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build_library(verbose=True, force="--force" in sys.argv))
