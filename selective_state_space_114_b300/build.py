"""Build libselscan.so in-tree with nvcc for sm_103a (B300).

    python selective_state_space_114_b300/build.py [--verbose]

(run as a file: importing the package itself loads the built library).

Compiles every csrc/*.cu into one shared library next to this file,
linked against the shared CUDA runtime (the same libcudart.so.13 that
PyTorch loads, so both share one runtime instance).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
SO = os.path.join(HERE, "libselscan.so")
# pipe-rate microbenchmark the bench uses for its ALU roofline denominators
PROBE_SRC = os.path.join(HERE, "probe", "pipes.cu")
PROBE_SO = os.path.join(HERE, "libssprobe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [os.path.join(INCLUDE, "selscan.h")]


def stale() -> bool:
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    return any(os.path.getmtime(p) > t for p in deps())


def build_probe(force: bool = False) -> str:
    if not force and os.path.exists(PROBE_SO) and \
            os.path.getmtime(PROBE_SO) >= os.path.getmtime(PROBE_SRC):
        return PROBE_SO
    tmp = PROBE_SO + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC",
           "--cudart", "shared", "-o", tmp, PROBE_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, PROBE_SO)
    return PROBE_SO


def build(force: bool = False, verbose: bool = False) -> str:
    build_probe(force)
    if not force and not stale():
        return SO
    # one object per source, compiled in parallel, then one link
    from concurrent.futures import ThreadPoolExecutor
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if verbose:
        flags.append("-Xptxas=-v")

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + f".{os.getpid()}.o")
        r = subprocess.run([nvcc(), *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    errs = [src + ":\n" + r.stdout + r.stderr for src, _, r in results if r.returncode != 0]
    if verbose:
        for _, _, r in results:
            sys.stderr.write(r.stdout + r.stderr)
    objs = [obj for _, obj, _ in results]
    try:
        if errs:
            raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
        tmp = SO + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc(), *ARCH, "--shared", "--cudart", "shared", "-o", tmp, *objs],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, SO)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return SO


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
