"""Build libepq.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into an object file under
``nvfp4_quantization_gb300/_build/``, then linked into one shared library.
FP contraction is disabled (``-fmad=false``) because the columnwise
re-quantisation is specified as separately rounded FP32 operations; explicit
fused multiply-adds in the kernels are unaffected.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = BUILD / "libepq.so"
SOURCES = ["api.cu", "route.cu", "route_noalloc.cu", "pack.cu", "unpack.cu", "receive.cu", "colwise_bf16.cu"]
HEADERS = ["epq_device.cuh", "epq_internal.h"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.environ.get("NVCC") or "/usr/local/cuda/bin/nvcc"
    return cand if os.path.exists(cand) else "nvcc"


def _flags(verbose: bool) -> list[str]:
    f = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale() -> bool:
    if not LIB.exists():
        return True
    deps = [CSRC / s for s in SOURCES + HEADERS] + [PKG.parent / "include" / "epq.h", Path(__file__)]
    return max(d.stat().st_mtime for d in deps) > LIB.stat().st_mtime


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and not _stale():
        return LIB
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [cc, *_flags(verbose), "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return str(obj)

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = BUILD / f"libepq.{os.getpid()}.so"
    cmd = [cc, ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
