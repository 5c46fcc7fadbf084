"""Build libw8a16.so in-tree with nvcc for sm_103a (GB300).

Usage: ``python -m fp8_weight_only_gemm_gb300.build`` or ``build_library()``.
Each CUDA translation unit compiles in parallel to an object; one link step
makes ``fp8_weight_only_gemm_gb300/_build/libw8a16.so``. A stamp of the
sources' hash and the flags skips rebuilding when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = BUILD / "libw8a16.so"

SOURCES = ["w8a16_api.cu", "w8a16_simt.cu", "w8a16_tc.cu", "w8a16_tc8.cu", "w8a16_w8a8.cu",
           "w8a16_quant.cu", "w8a16_gemv.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libw8a16.so")


def _stamp() -> str:
    h = hashlib.sha256()
    for p in sorted(list(CSRC.glob("*")) + [INCLUDE / "w8a16.h", Path(__file__)]):
        if p.is_file():
            h.update(p.name.encode())
            h.update(p.read_bytes())
    h.update(" ".join(ARCH + FLAGS).encode())
    h.update(platform.machine().encode())      # never reuse a build from another host arch
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False) -> Path:
    BUILD.mkdir(parents=True, exist_ok=True)
    stamp_file = BUILD / "stamp"
    stamp = _stamp()
    if not force and LIB.exists() and stamp_file.exists() and stamp_file.read_text() == stamp:
        return LIB
    nvcc = _nvcc()
    inc = ["-I", str(INCLUDE), "-I", str(CSRC)]

    def compile_one(src: str) -> tuple[str, str]:
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *inc, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return str(obj), r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = "\n".join(err for _, err in results)
    (BUILD / "ptxas.log").write_text(log)
    if verbose:
        print(log)
    tmp = BUILD / f"libw8a16.so.tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *[o for o, _ in results], "-lcudart_static",
           "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    stamp_file.write_text(stamp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build_library(force="--force" in sys.argv, verbose=True))
