"""Build libwql.so in-tree with nvcc for sm_103a (no CMake, no setuptools).

Each ``csrc/*.cu`` translation unit is compiled in parallel to an object file, then linked into
``weight_quantized_linear_gb300/_build/libwql.so``.  Rebuilds only what changed (source or any
header newer than the object).  ``build(trace=True)`` makes the developer build with the W4A16
kernels' phase stamps (``-DWQL_PHASE_TRACE``) in ``_build_trace/`` instead; the package loads the
default build unless told otherwise.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libwql.so")
TRACE_OUT_DIR = os.path.join(PKG, "_build_trace")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                     "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src: str, obj: str, extra: list[str], defines: list[str]) -> None:
    cmd = [_nvcc()] + NVCC_FLAGS + defines + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if extra:
        sys.stderr.write(r.stderr)


def build(force: bool = False, verbose_ptxas: bool = False, trace: bool = False) -> str:
    out_dir = TRACE_OUT_DIR if trace else OUT_DIR
    lib = os.path.join(out_dir, "libwql.so")
    defines = ["-DWQL_PHASE_TRACE"] if trace else []
    os.makedirs(out_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _headers_mtime()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(out_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or verbose_ptxas or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), hdr_t):
            jobs.append((s, o))
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda so: _compile(so[0], so[1], extra, defines), jobs))
    if force or jobs or not os.path.exists(lib):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, trace="--trace" in sys.argv))
