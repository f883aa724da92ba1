"""Build libkpool.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery).  Translation units compile in parallel."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkpool.so")
SOURCES = ["kpool_api.cu", "kpool_compress.cu", "kpool_expand.cu", "kpool_score.cu",
           "kpool_pipeline.cu", "kpool_project.cu", "kpool_mla.cu"]
HEADERS = ["kpool_internal.h", "kpool_ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    nv = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nv):
        raise RuntimeError("nvcc not found")
    return nv


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """variant "" builds libkpool.so; "phase_timers" builds libkpool_phase_timers.so with
    -DKPOOL_PHASE_TIMERS (per-phase cycle counters of the scoring kernel)."""
    build_dir, lib_path = BUILD, LIB
    if variant:
        extra_flags = tuple(extra_flags) + ("-DKPOOL_%s" % variant.upper(),)
        build_dir = os.path.join(HERE, "_build_" + variant)
        lib_path = os.path.join(HERE, "libkpool_%s.so" % variant)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS]
    hdrs.append(os.path.join(os.path.dirname(HERE), "include", "kpool.h"))

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
            if verbose and r.stderr:
                print(r.stderr, file=sys.stderr)
        return o

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    var = ""
    for a in sys.argv[1:]:
        if a.startswith("--variant="):
            var = a.split("=", 1)[1]
    print(build(force="--force" in sys.argv, verbose=True, variant=var))
