"""Builds libmhc.so in-tree for sm_103a: one nvcc process per translation unit, in parallel,
then one link. No cmake, no setuptools; a few seconds per file."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmhc.so")
SOURCES = ["fused.cu", "small.cu", "abi.cu", "host_pipeline.cu"]
HEADERS = ["ptx.cuh", "mix_math.cuh", "hc_arith.cuh", "internal.h", "layout.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: a separate float32 multiply and add must stay two roundings (hc_post and hc_pre
# are defined with float32 products and float32 sums; their kernels also spell the products and
# sums out as explicit round-to-nearest PTX); explicit fma instructions are unaffected.
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xptxas=--fmad=false",
          "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
          f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _newest_input_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "mhc.h"),
                                                                  os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libmhc.so if any source is newer than it. Returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input_mtime():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *CFLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           f"-Xlinker=-rpath,{libdir}", f"-L{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
