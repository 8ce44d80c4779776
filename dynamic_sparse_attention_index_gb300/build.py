"""Compile the CUDA library (libvs.so) in-tree for sm_103a.

nvcc compiles every ``csrc/*.cu`` in parallel into ``_build/`` and links a
shared library next to this file.  Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libvs.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


STAMP = os.path.join(BUILD, "flags.txt")


def _flags() -> list:
    # VS_WAIT_PROFILE=1..6 compiles in the attention kernels' wait-cycle
    # counters (all, dK/dV only, query-major only, MMA issue of dK/dV or
    # query-major only)
    mode = os.environ.get("VS_WAIT_PROFILE", "")
    extra = [f"-DVS_WAIT_PROFILE={mode}"] if mode in ("1", "2", "3", "4", "5", "6", "7", "8") else []
    # VS_DEBUG=1: device bounds checks (VS_ERR_BOUNDS in the status word)
    if os.environ.get("VS_DEBUG", "") == "1":
        extra.append("-DVS_DEBUG=1")
    return FLAGS + extra


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    try:
        with open(STAMP) as f:
            if f.read() != " ".join(_flags()):
                return True
    except OSError:
        return True
    t = os.path.getmtime(LIB)
    deps = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *_flags(), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    # a shared library links with unresolved symbols; refuse any of our own
    r = subprocess.run(["nm", "-u", "-C", tmp], capture_output=True, text=True)
    missing = [l for l in r.stdout.splitlines() if "vs::" in l]
    if missing:
        os.remove(tmp)
        raise RuntimeError("unresolved library symbols:\n" + "\n".join(missing))
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(" ".join(_flags()))
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, force=True))
