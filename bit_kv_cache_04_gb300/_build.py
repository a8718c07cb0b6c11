"""Builds libkvq.so in-tree with nvcc for sm_103a (GB300)."""

from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")
# The bounds-checked variant (every computed cache address checked against
# its buffer segment, misses recorded as KVQ_DEV_BOUNDS): a test build.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libkvq_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]

# (source, extra flags).  The append path quantizes with a fixed fp32 op
# order, so it is compiled without FMA contraction.
SOURCES = [
    ("kvq_api.cu", []),
    ("append.cu", ["--fmad=false"]),
    ("append_fast.cu", ["--fmad=false"]),
    ("append_fast_zp_f16.cu", ["--fmad=false"]),
    ("append_fast_zp_bf16.cu", ["--fmad=false"]),
    ("append_rot.cu", ["--fmad=false"]),
    ("decode_generic.cu", []),
    ("decode_mma.cu", []),
    ("decode_step.cu", []),
    ("decode_step_kivi.cu", []),
    ("decode_step_d128.cu", []),
    ("decode_step_d256.cu", []),
    ("dequant.cu", []),
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles every translation unit in parallel and links libkvq.so (or,
    with checked=True, the bounds-checked libkvq_checked.so).  Returns the
    library path."""
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    flags = ["-DKVQ_BOUNDS_CHECK"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "kvq.h"))

    def compile_one(item):
        src, extra = item
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        srcp = os.path.join(CSRC, src)
        if not force and _newer(obj, [srcp] + headers):
            return obj
        cmd = [nvcc, *ARCH, *COMMON, *flags, *extra, "-c", srcp, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or not _newer(lib, objs):
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
