"""Build libattn.so in-tree with nvcc for sm_103a (no CMake, no setuptools).

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file
under ``_build/``; the objects link into ``libattn.so`` next to this file
with the CUDA runtime linked statically, so the library loads into any
process (PyTorch's or a plain C program) without a torch ABI dependency.
Run ``python -m exact_scaled_dot_flash_gb300.build`` or call :func:`build`.

``build(checked=True)`` (``python -m exact_scaled_dot_flash_gb300.build
--checked``) makes the bounds-checked variant ``libattn_checked.so`` from the
same sources with ``-DATTN_CHECKED`` (objects under ``_build_checked/``): its
paged, MLA, split and backward kernels test every computed global and
shared-memory index and record a violation in the device status word
(ATTN_STATUS_BOUNDS) instead of making the access.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")
CHECKED_OUT_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(PKG, "libattn_checked.so")
CHECKED_FLAGS = ("-DATTN_CHECKED",)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _digest(paths, extra=()):
    h = hashlib.sha256()
    for p in paths:
        h.update(os.path.basename(p).encode())  # not the directory: the same on every machine
        with open(p, "rb") as f:
            h.update(f.read())
    for e in extra:
        h.update(str(e).encode())
    return h.hexdigest()


def kernel_source_digest(names=None) -> str:
    """Digest of the CUDA sources and headers a kernel is built from (file names
    under csrc/ or include/; every source and header when None): identifies the
    kernels a profile describes."""
    if names is None:
        paths = _sources() + _headers()
    else:
        paths = [os.path.join(CSRC, n) if os.path.exists(os.path.join(CSRC, n)) else os.path.join(INCLUDE, n)
                 for n in sorted(names)]
    return _digest(paths)[:16]


def _compile(src, hdr_digest, verbose, extra_flags, out_dir=OUT_DIR):
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    stamp = obj + ".sha"
    key = _digest([src], (hdr_digest, *NVCC_FLAGS, *extra_flags))
    if os.path.exists(obj) and os.path.exists(stamp) and open(stamp).read() == key:
        return obj, ""
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    with open(stamp, "w") as f:
        f.write(key)
    return obj, r.stdout + r.stderr


def build(verbose: bool = False, jobs: int | None = None, extra_flags=(), checked: bool = False) -> str:
    """Compile every CUDA translation unit for sm_103a and link libattn.so
    (with ``checked``, the bounds-checked libattn_checked.so)."""
    out_dir, lib = (CHECKED_OUT_DIR, CHECKED_LIB) if checked else (OUT_DIR, LIB)
    if checked:
        extra_flags = tuple(extra_flags) + CHECKED_FLAGS
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    hdr = _digest(_headers())
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        futs = [ex.submit(_compile, s, hdr, verbose, tuple(extra_flags), out_dir) for s in srcs]
        objs = []
        for f in futs:
            o, log = f.result()
            objs.append(o)
            if log:
                logs.append(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        sys.stdout.write("".join(logs))
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checked="--checked" in sys.argv))
