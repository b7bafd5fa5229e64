"""Build the CUDA library in-tree: dense_gemm_sgemm_gb300/_build/libgemm_gb300.so.

Every translation unit under csrc/ is compiled for sm_103a only (tcgen05 and the other
arch-specific features need the `a` target), in parallel, and linked into one shared
library with the static CUDA runtime.  No fast-math: denormals, IEEE division and square
root stay on, which the strict-FP32 path relies on.

    python -m dense_gemm_sgemm_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libgemm_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the library needs the CUDA 13 toolkit")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h"))) + sorted(
        glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(ROOT, "include", "gemm_gb300.h"),
                                                   os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(nvcc, src, obj, ptxas_verbose):
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include"),
           "-c", src, "-o", obj]
    if ptxas_verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    if not force and not ptxas_verbose and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = []
        for src in _sources():
            obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            futs.append(ex.submit(_compile, nvcc, src, obj, ptxas_verbose))
        for f in futs:
            src, rc, log = f.result()
            if rc != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{log}")
            if log.strip() and (ptxas_verbose or not quiet):
                print(f"--- {os.path.basename(src)}\n{log}", file=sys.stderr)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    # Static CUDA runtime; driver entry points (tensor-map encoding) are looked up at run
    # time through cudaGetDriverEntryPointByVersion, so the library loads without a driver.
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, ptxas_verbose=a.verbose_ptxas, quiet=False))


if __name__ == "__main__":
    main()
