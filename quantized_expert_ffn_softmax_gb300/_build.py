"""Builds libmoe_gb300.so (the C-ABI library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libmoe_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    return os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "moe.h"), __file__]


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    with open(LIB + ".lock", "w") as lf:
        fcntl.flock(lf, fcntl.LOCK_EX)
        try:
            newest = max(os.path.getmtime(p) for p in _deps())
            if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
                return LIB
            objs = []

            def compile_one(src):
                obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
                cmd = [_nvcc(), *ARCH, *FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src,
                       "-o", obj]
                r = subprocess.run(cmd, capture_output=True, text=True)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
                if verbose:
                    print(r.stdout + r.stderr)
                return obj

            with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
                objs = list(ex.map(compile_one, _sources()))
            tmp = LIB + ".tmp%d" % os.getpid()
            cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
            os.replace(tmp, LIB)
        finally:
            fcntl.flock(lf, fcntl.LOCK_UN)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, force=True))
