"""Build libpkv.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to ``_build/*.o`` and
linked into ``paged_kv_decode_bind_gb300/libpkv.so`` (static cudart, so the
library loads without a CUDA runtime on the loader path).  A unit is rebuilt
when it or any header is newer than its object.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + os.path.join(ROOT, "include")]


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(obj, src, hdr_mtime):
    return not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_mtime)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile every kernel unit and link libpkv.so; returns the library path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    if not os.path.exists(LIB):
        force = True  # objects left from another machine are never trusted
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    jobs = []
    for s in srcs:
        obj = os.path.join(OUT_DIR, os.path.basename(s)[:-3] + ".o")
        if force or ptxas_info or _stale(obj, s, hdr):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", s, "-o", obj]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append((s, cmd))

    def run(job):
        s, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r

    failed = []
    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for s, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                failed.append(os.path.basename(s))
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    objs = [os.path.join(OUT_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if force or jobs or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv,
                force="--force" in sys.argv))
