"""Build ``libbwgemm.so`` in-tree (``_build/``) with nvcc for sm_103a.

One ``-gencode`` (``arch=compute_103a,code=sm_103a``), translation units
compiled in parallel, statically linked CUDA runtime.  ``python -m
dense_gemm_blackwell_03_gb300.build [--force] [--verbose]`` runs it by hand.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libbwgemm.so")

SOURCES = ["gemm_sm103.cu", "skinny_sm103.cu", "wholek_sm103.cu", "api.cpp", "planner.cpp", "noalloc.cu", "probe.cu",
           "microbench.cu"]
HEADERS = ["ptx.cuh", "gemm_kernel.cuh", "skinny_kernel.cuh", "wholek_kernel.cuh", "kernel_params.h", "internal.h", "tuned_table.h"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libbwgemm")
    return found


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "bwgemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(nvcc: str, src: str, obj: str, verbose: bool):
    cmd = [nvcc, *GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return res.stderr if verbose else ""


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of ``libbwgemm.so``."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tag = f"{os.getpid()}"
    objs = [os.path.join(OUT_DIR, f"{os.path.splitext(s)[0]}.{tag}.o") for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(lambda so: _compile(nvcc, so[0], so[1], verbose), zip(SOURCES, objs)))
    if verbose:
        for s, log in zip(SOURCES, logs):
            if log:
                print(f"--- {s}\n{log}", file=sys.stderr)
    tmp = f"{LIB_PATH}.{tag}.tmp"
    cmd = [nvcc, *GENCODE, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        if os.path.exists(o):
            os.remove(o)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    main()
