"""Build libclcgemm.so in-tree: one nvcc compile per translation unit (in parallel),
then a shared-library link.  sm_103a only; the CUDA runtime is linked statically so the
library loads on machines without a GPU (compute calls then fail with an error code).

``--checked`` builds libclcgemm_checked.so instead: the same sources compiled with
CLCG_BOUNDS_CHECK, whose kernels check every tile coordinate against its problem before
using it, record a failure in the device error word (gemm_sync then returns
GEMM_ERR_BOUNDS) and skip the tile; nothing traps.  The binding loads it when the
environment sets CLCGEMM_CHECKED=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libclcgemm.so")
BUILD_DIR = os.path.join(PKG, "_build")
OUT_CHECKED = os.path.join(PKG, "libclcgemm_checked.so")
BUILD_DIR_CHECKED = os.path.join(PKG, "_build_checked")
SOURCES = ["api.cu", "kern_n128_c1.cu", "kern_n256_c1.cu", "kern_n256_c2.cu", "kern_n256_c2mc.cu", "kern_n256_c4mc.cu", "kern_n256_c2x2.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "clcgemm.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, checked: bool = False) -> str:
    out = OUT_CHECKED if checked else OUT
    build_dir = BUILD_DIR_CHECKED if checked else BUILD_DIR
    if not force and os.path.exists(out) and os.path.getmtime(out) >= _newest_input():
        return out
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checked:
        extra += ["-DCLCG_BOUNDS_CHECK"]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if ptxas_info or verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static", "-Xlinker", "--exclude-libs,ALL"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked="--checked" in sys.argv))
