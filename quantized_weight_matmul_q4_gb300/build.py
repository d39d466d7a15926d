"""Builds libkq.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel to an object file, then linked
into ``_lib/libkq.so`` (CUDA runtime linked statically). A unit is rebuilt only
when its source or a header is newer than its object file.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
OUT_DIR = os.path.join(PKG_DIR, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libkq.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["kq_api.cu", "kq_quant.cu", "kq_matvec.cu", "kq_gemm.cu", "kq_gemm_noalloc.cu", "kq_combine.cu", "kq_tq4.cu"]
# A measurement aid outside libkq (the tensor-core MMA issue rate), in a library of its own.
PROBE_SOURCES = ["probe_mma.cu"]
PROBE_LIB_PATH = os.path.join(OUT_DIR, "libkqprobe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkq")


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "kq.h"))
    return hs


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, extra) -> None:
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compiles every source and links libkq.so; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    hdrs = _headers()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    objs = []
    probe_objs = [os.path.join(OUT_DIR, s.replace(".cu", ".o")) for s in PROBE_SOURCES]
    for s in PROBE_SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(OUT_DIR, s.replace(".cu", ".o"))
        if ptxas_info or _stale(obj, [src, *hdrs]):
            jobs.append((src, obj))
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(OUT_DIR, s.replace(".cu", ".o"))
        objs.append(obj)
        if ptxas_info or _stale(obj, [src, *hdrs]):
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(_compile, s, o, extra) for s, o in jobs]
            for f in futs:
                f.result()
    for path, parts in ((LIB_PATH, objs), (PROBE_LIB_PATH, probe_objs)):
        if _stale(path, parts):
            tmp = path + ".tmp"
            cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *parts, "-Xcompiler", "-fPIC"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, path)
    if verbose:
        print(f"libkq: {LIB_PATH} ({len(jobs)} unit(s) rebuilt)")
    return LIB_PATH


if __name__ == "__main__":
    import sys
    build(verbose=True, ptxas_info="--ptxas-info" in sys.argv)
