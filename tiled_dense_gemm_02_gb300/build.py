"""Build libtgemm.so in-tree with nvcc for sm_103a (no GPU needed to compile).

    python tiled_dense_gemm_02_gb300/build.py [--force] [-v]

This file is standalone: it is run or loaded by path (``load()`` below), never
imported through the package, whose import needs the built library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(HERE, "libtgemm.so")
# the FP32 FMA-throughput probe the benchmark uses for the SIMT roofline (not part of libtgemm.so)
PROBE_SOURCE = os.path.join(CSRC, "probe", "fp32_peak.cu")
PROBE_LIBRARY = os.path.join(HERE, "libtgemm_probe.so")
HEADER = os.path.join(ROOT, "include", "tgemm.h")

NVCC = os.environ.get("NVCC", "nvcc")
NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def load():
    """This module, loaded by file path without importing the package."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("tgemm_build", os.path.abspath(__file__))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def inputs() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + sorted(glob.glob(os.path.join(CSRC, "*.inc"))) + \
        [HEADER, os.path.abspath(__file__)]


def stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(p) > t for p in inputs())


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build_probe(force: bool = False) -> str:
    """Compile the FP32 FMA-throughput probe into its own shared library."""
    if not force and os.path.exists(PROBE_LIBRARY) and \
            os.path.getmtime(PROBE_LIBRARY) >= max(os.path.getmtime(PROBE_SOURCE), os.path.getmtime(__file__)):
        return PROBE_LIBRARY
    tmp = PROBE_LIBRARY + ".tmp"
    cmd = [NVCC, *NVCC_FLAGS, "-shared", "-o", tmp, PROBE_SOURCE]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {PROBE_SOURCE}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, PROBE_LIBRARY)
    return PROBE_LIBRARY


def build(force: bool = False, extra: list[str] | None = None) -> str:
    """Compile every CUDA source in parallel and link the shared library (and
    the FP32 probe beside it)."""
    build_probe(force)
    if not force and not stale():
        return LIBRARY
    os.makedirs(OBJ_DIR, exist_ok=True)
    extra = extra or []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources()), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), sources()))
    tmp = LIBRARY + ".tmp"
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, extra=["-Xptxas", "-v"] if "-v" in sys.argv else None))
