"""Build the CUDA library (libmoeffn.so) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library under ``_build/<machine>/``.  A stamp of the sources and
flags skips rebuilds when nothing changed.  ``variant="bounds"`` builds
libmoeffn_bounds.so with MOEFFN_BOUNDS_CHECK (device index checks that report
through the status word; for tests).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["api.cu", "layout_kernels.cu", "gemm_kernels.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "kernels.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


VARIANTS = {"": [], "bounds": ["-DMOEFFN_BOUNDS_CHECK"]}


def lib_path(variant: str = "") -> str:
    name = "libmoeffn.so" if not variant else f"libmoeffn_{variant}.so"
    return os.path.join(HERE, "_build", platform.machine(), name)


def _digest(flags) -> str:
    h = hashlib.sha256()
    for f in SOURCES + HEADERS:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(INCLUDE, "moeffn.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(ARCH + flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    so = lib_path(variant)
    flags = FLAGS + VARIANTS[variant]
    out = os.path.join(os.path.dirname(so), variant or "product")
    os.makedirs(out, exist_ok=True)
    digest = _digest(flags)
    stamp = so + ".stamp"
    if not force and os.path.exists(so) and os.path.exists(stamp) and open(stamp).read().strip() == digest:
        return so

    def compile_one(src: str) -> str:
        obj = os.path.join(out, src.replace(".cu", ".o"))
        cmd = [nvcc()] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = so + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, so)
    with open(stamp, "w") as f:
        f.write(digest)
    return so


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
