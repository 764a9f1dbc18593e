"""Build libdcp.so (sm_103a) in-tree with nvcc: one object per .cu, compiled
in parallel, then linked into a shared library next to this file."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdcp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources(d):
    return sorted(os.path.join(d, f) for f in os.listdir(d) if f.endswith(".cu"))


def _headers(d):
    return [os.path.join(d, f) for f in os.listdir(d) if f.endswith((".cuh", ".h"))]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, obj, extra=()):
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr


def build_library(lib=LIB, srcdir=CSRC, name="dcp", verbose=False, extra=()) -> str:
    """Compile and link one shared library from the .cu files of srcdir."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources(srcdir)
    deps = srcs + _headers(srcdir) + _headers(os.path.join(ROOT, "include")) + [__file__]
    if not _stale(lib, deps):
        return lib
    objs = [os.path.join(BUILD, f"{name}_{os.path.basename(s)[:-3]}.o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], extra), zip(srcs, objs)))
    if verbose:
        for s, log in zip(srcs, logs):
            if log.strip():
                print(os.path.basename(s), log, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt",
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(verbose=False):
    out = [build_library(verbose=verbose)]
    synth_dir = os.path.join(ROOT, "workloads")
    out.append(build_library(os.path.join(synth_dir, "libdcp_synth.so"), synth_dir, "synth",
                             verbose=verbose))
    return out


if __name__ == "__main__":
    for p in build_all(verbose="-v" in sys.argv):
        print(p)
