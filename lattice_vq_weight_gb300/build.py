"""Build liblq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into a shared
library with the CUDA runtime linked statically, so the library loads without
a driver (symbol checks on CPU-only hosts) and uses the caller's streams.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "liblq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ("lq_api.cu", "lq_quantize.cu", "lq_quantize_fmt.cu", "lq_quantize_dither.cu", "lq_gemv.cu", "lq_gemm.cu",
           "lq_rice.cu", "lq_calib.cu", "lq_kv.cu", "lq_kv_dither.cu", "lq_kv_rice.cu")
# Objects: one per source, except lq_kv_rice.cu, compiled once per (lattice,
# norm format) pair so that its slow instantiations build in parallel.
UNITS = tuple((s, s.replace(".cu", ".o"), ()) for s in SOURCES if s != "lq_kv_rice.cu") + tuple(
    ("lq_kv_rice.cu", f"lq_kv_rice_{p}.o", (f"-DLQ_KV_RICE_PART={p}",)) for p in range(8))


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblq")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "lq.h"))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj, *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every source into liblq.so; returns the library path."""
    if not force and not is_stale():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs = []
    # the slowest units first, so that they start before the pool fills
    order = sorted(UNITS, key=lambda u: (u[0] != "lq_kv_rice.cu", u[1]))
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        futs = {}
        for s, o, defs in order:
            obj = os.path.join(BUILD_DIR, o)
            objs.append(obj)
            futs[ex.submit(_compile, nvcc, os.path.join(CSRC, s), obj, list(defs) + list(extra_flags))] = o
        for f in cf.as_completed(futs):
            log = f.result()
            if verbose and log:
                print(log, file=sys.stderr)
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
