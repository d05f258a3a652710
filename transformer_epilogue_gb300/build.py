"""Build the in-tree C-ABI library ``lib/libtransformer_epilogue.so`` with nvcc.

One translation unit per op family, compiled in parallel for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), then linked into a shared
library with the CUDA runtime linked statically.  Objects go to ``_build/``;
a source newer than its object (or a changed header) triggers a rebuild.

Usage:  python -m transformer_epilogue_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libtransformer_epilogue.so")

SOURCES = ["ep_api.cpp", "skip_layer_norm.cu", "bias_softmax.cu", "elementwise.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build the library)")


def _headers_mtime() -> float:
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, force: bool, verbose: bool, extra: list, build_dir: str = BUILD) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(build_dir, src + ".o")
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(path), _headers_mtime()):
        return obj
    cmd = [nvcc(), "-c", path, "-o", obj] + ARCH + COMMON + extra
    if src.endswith(".cu"):  # the three kernel files compile side by side; each splits its optimizer over cores
        cmd += ["-split-compile", str(max(1, (os.cpu_count() or 3) // 3))]
    if verbose:
        print(" ".join(cmd), flush=True)
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    if verbose and (p.stdout or p.stderr):
        print(p.stdout + p.stderr, flush=True)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          defines: dict | None = None, out_dir: str | None = None) -> str:
    """Build the library; returns its path.  ``defines`` (name -> value) are
    passed as -D flags (the tuning constants of csrc/tuning.h); with
    ``out_dir`` the objects and library go there instead of the package."""
    build_dir = BUILD if out_dir is None else os.path.join(out_dir, "_build")
    lib = LIB if out_dir is None else os.path.join(out_dir, os.path.basename(LIB))
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    extra += [f"-D{k}={v}" for k, v in (defines or {}).items()]
    force = force or bool(defines)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force or ptxas_verbose, verbose or ptxas_verbose, extra, build_dir),
                           SOURCES))
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, lib)
    return lib


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true", help="print registers/spills per kernel")
    args = ap.parse_args(argv)
    print(build(args.force, args.verbose, args.ptxas_verbose))
    return 0


if __name__ == "__main__":
    sys.exit(main())
