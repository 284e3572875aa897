"""In-tree build of the package's native libraries with nvcc for sm_103a.

``libkvpool.so``  -- the two-pool KV cache: host runtime (C++) + CUDA kernels.
``gen/libkvgen.so`` -- the seeded synthetic-input generator (host + device).

Objects are compiled in parallel under ``_build/`` and linked with the static
CUDA runtime.  A library is rebuilt only when one of its sources or headers is
newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
           "--expt-relaxed-constexpr", "-Xptxas", "-O3"]

_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build heterogeneous_compressed_kv_gb300")


LIBS = {
    "kvpool": {
        "out": os.path.join(PKG, "libkvpool.so"),
        "sources": ["csrc/kvpool_host.cpp", "csrc/kvpool_append.cu", "csrc/kvpool_score.cu", "csrc/kvpool_select.cu",
                    "csrc/kvpool_attend.cu", "csrc/kvpool_image.cu"],
        "headers": ["csrc/kvpool_internal.h", "csrc/device_util.cuh", "../include/kvpool.h"],
    },
    "kvgen": {
        "out": os.path.join(PKG, "gen", "libkvgen.so"),
        "sources": ["gen/kvgen_host.c", "gen/kvgen_device.cu"],
        "headers": ["gen/kvgen.h"],
    },
}


def _stale(out, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.exists(d) and os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, extra) -> None:
    cmd = [nvcc()] + ARCH + NVFLAGS + ["-I", INCLUDE, "-I", os.path.join(PKG, "csrc"), "-I",
                                       os.path.join(PKG, "gen")] + extra + ["-c", src, "-o", obj]
    if src.endswith(".c"):
        # plain C host file: compile as C11 with the host compiler
        cmd = [nvcc(), "-O3", "-Xcompiler", "-fPIC", "-Xcompiler", "-std=c11", "-Xcompiler",
               "-ffp-contract=off", "-I", os.path.join(PKG, "gen"), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")


def build_lib(name: str, force: bool = False, extra=()) -> str:
    spec = LIBS[name]
    srcs = [os.path.join(PKG, s) for s in spec["sources"]]
    hdrs = [os.path.normpath(os.path.join(PKG, h)) for h in spec["headers"]]
    out = spec["out"]
    with _lock:
        if not force and not _stale(out, srcs + hdrs + [__file__]):
            return out
        os.makedirs(BUILD, exist_ok=True)
        objs = [os.path.join(BUILD, f"{name}_{os.path.basename(s)}.o") for s in srcs]
        with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
            list(ex.map(lambda so: _compile(so[0], so[1], list(extra)), zip(srcs, objs)))
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return out


def build_all(force: bool = False) -> None:
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda n: build_lib(n, force), list(LIBS)))
