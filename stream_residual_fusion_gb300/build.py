"""Builds libmhc.so in-tree for sm_103a: one nvcc process per translation unit, in parallel,
then one link. No cmake, no setuptools; a few seconds per file.

build(checked=True) builds the same sources with MHC_CHECKED=1 into libmhc_checked.so: every
copy, store and exchange access of the fused step tests its index first, skips a failing one and
reports it through mhc_get_status (MHC_ERR_BOUNDS). build_all() builds both at once."""
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
LIB_CHECKED = os.path.join(PKG, "libmhc_checked.so")
SOURCES = ["fused.cu", "cluster.cu", "small.cu", "abi.cu", "host_pipeline.cu", "backward.cu"]
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


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile and link libmhc.so (libmhc_checked.so with checked=True) if any source is newer
    than it. Returns its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input_mtime():
        return lib
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    defs = ["-DMHC_CHECKED=1"] if checked else []

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *CFLAGS, *defs, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
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
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           f"-Xlinker=-rpath,{libdir}", f"-L{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False, verbose: bool = False) -> list[str]:
    """The regular and the bounds-checked library, built at the same time."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        jobs = [ex.submit(build, force, verbose, (), c) for c in (False, True)]
        return [j.result() for j in jobs]


if __name__ == "__main__":
    print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
