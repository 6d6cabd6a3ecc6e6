"""In-tree build of libinjectscale.so (and the synthetic-input generator) for sm_103a.

Plain nvcc, one translation unit per process in parallel, static CUDA runtime,
so the shared object depends on nothing but libc/libstdc++ and the driver it
finds at run time.  ``build()`` skips the work when every output is newer
than every source.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libinjectscale.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "csrc", "synthgen.cu")
SYNTH_LIB = os.path.join(ROOT, "synth", "lib", "libsynthgen.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]
SOURCES = ["store.cu", "retrieve.cu", "inject.cu", "simgemm.cu", "capture.cu"]
HEADERS = [os.path.join(INCLUDE, "injectscale.h")] + [
    os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str], verbose: bool) -> None:
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, file=sys.stderr)


def build(verbose: bool = False, force: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile libinjectscale.so and libsynthgen.so if stale; return the library path."""
    flags = NVCC_FLAGS + list(extra_flags or [])
    os.makedirs(LIB_DIR, exist_ok=True)
    os.makedirs(os.path.dirname(SYNTH_LIB), exist_ok=True)
    obj_dir = os.path.join(LIB_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    nv = nvcc()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    objs = [os.path.join(obj_dir, s.replace(".cu", ".o")) for s in SOURCES]
    jobs = []
    for src, obj in zip(srcs, objs):
        if force or extra_flags or _stale(obj, [src] + HEADERS):
            jobs.append([nv] + flags + ["-c", src, "-o", obj])
    synth_job = None
    if force or _stale(SYNTH_LIB, [SYNTH_SRC]):
        synth_job = [nv] + ARCH + ["-O3", "-Xcompiler", "-fPIC", "-shared", SYNTH_SRC, "-o", SYNTH_LIB]
    with ThreadPoolExecutor(max_workers=len(jobs) + 1) as ex:
        futs = [ex.submit(_run, j, verbose) for j in jobs]
        if synth_job:
            futs.append(ex.submit(_run, synth_job, verbose))
        for f in futs:
            f.result()
    if jobs or _stale(LIB, objs):
        _run([nv] + ARCH + ["-shared", "-Xlinker", "--no-undefined", "-o", LIB] + objs, verbose)
    return LIB


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)
    print(LIB)
