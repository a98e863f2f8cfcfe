"""Build libllm.so in-tree for sm_103a: one nvcc per translation unit, in parallel, then a link.

    python -m transformer_decode_kv_gb300.build [--force] [--verbose]

Objects go to transformer_decode_kv_gb300/_build/; the library to
transformer_decode_kv_gb300/libllm.so. A source is recompiled when it or a header is newer than
its object.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libllm.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _flags(extra=()):
    return (ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O3",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
            + list(extra))


def _stale(src: str, obj: str, headers) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or any(os.path.getmtime(h) > t for h in headers)


def build(force: bool = False, verbose: bool = False, jobs: int = 0) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    cc = nvcc()
    todo = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s) + ".o")
        objs.append(o)
        if force or _stale(s, o, headers):
            todo.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [cc] + _flags(["-Xptxas", "-v"] if verbose else []) + ["-c", s, "-o", o]
        if s.endswith(".cpp"):
            cmd = [cc] + _flags() + ["-x", "c++", "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return s, r.stderr

    if todo:
        n = jobs or min(len(todo), max(2, os.cpu_count() or 2))
        with cf.ThreadPoolExecutor(n) as ex:
            for s, err in ex.map(compile_one, todo):
                if verbose and err:
                    print(f"== {os.path.basename(s)}\n{err}", file=sys.stderr)
    if todo or not os.path.exists(LIB):
        cmd = [cc] + ARCH + ["-shared", "-o", LIB + ".tmp"] + objs + ["-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
