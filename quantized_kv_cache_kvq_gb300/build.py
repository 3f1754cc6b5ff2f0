"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel; the link step produces
``quantized_kv_cache_kvq_gb300/libkvq.so``.  Object files go to ``_build/``.
A unit is recompiled only when a source or header is newer than its object.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq")
    return cand


def _deps() -> list[str]:
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.inc")) + [
        os.path.join(PKG, "..", "include", "kvq.h")
    ]


def _compile(nvcc: str, src: str) -> tuple[str, int, str]:
    obj = os.path.join(OUT, os.path.basename(src)[:-3] + ".o")
    newest = max(os.path.getmtime(p) for p in [src] + _deps())
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest:
        return obj, 0, ""
    cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    with open(obj[:-2] + ".log", "w") as f:
        f.write(p.stdout + p.stderr)
    return obj, p.returncode, p.stdout + p.stderr


def build(verbose: bool = False) -> str:
    """Compile every CUDA unit and link libkvq.so; returns the library path."""
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s), srcs))
    bad = [(o, log) for o, rc, log in results if rc != 0]
    if bad:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"{o}:\n{log}" for o, log in bad))
    objs = [o for o, _, _ in results]
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", LIB, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    if verbose:
        for o, _, log in results:
            print(os.path.basename(o), log.strip()[:200])
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
