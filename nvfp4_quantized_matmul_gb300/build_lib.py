"""Build libnvfp4.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each translation unit compiles in parallel to an object under ``_build/``;
the objects link into ``nvfp4_quantized_matmul_gb300/libnvfp4.so``. A unit is
recompiled when its source, a header or the flags change.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libnvfp4.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]
SOURCES = ["nvfp4_api.cu", "nvfp4_stream.cu", "nvfp4_qmv.cu", "nvfp4_qmv_tma.cu", "nvfp4_qmv_stream.cu", "nvfp4_qmm_tc.cu",
           "nvfp4_qmv_nt.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _headers_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, os.path.join(ROOT, "include")):
        for name in sorted(os.listdir(d)):
            if name.endswith((".h", ".cuh")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + f.read())
    return h.hexdigest()


def _compile(src: str, extra: list[str], hdr: str, verbose: bool) -> str:
    path = os.path.join(CSRC, src)
    with open(path, "rb") as f:
        body = f.read()
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-c", path]
    key = hashlib.sha256(body + hdr.encode() + " ".join(cmd).encode()).hexdigest()[:16]
    obj = os.path.join(BUILD, f"{os.path.splitext(src)[0]}.{key}.o")
    if not os.path.exists(obj):
        tmp = obj + ".tmp"
        res = subprocess.run(cmd + ["-o", tmp], capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr.strip():
            print(res.stderr, file=sys.stderr)
        os.replace(tmp, obj)
    return obj


def build(verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile and link the library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra or [])
    hdr = _headers_digest()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, hdr, verbose), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []
    print(build(verbose=v or bool(extra), extra=extra))
