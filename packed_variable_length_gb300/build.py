"""Builds libpvl.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel to an object file
in csrc/../_build/, then nvcc links the shared library with the static CUDA
runtime.  The library depends only on the CUDA driver at run time; it finds
cuTensorMapEncodeTiled through the runtime's driver entry-point query, so it
loads on a machine without a GPU (every device call then fails cleanly).

Usage: python -m packed_variable_length_gb300.build [--force] [--verbose]
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpvl.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libpvl.so")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compiles csrc/*.cu and links libpvl.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    headers = _headers()
    todo = [s for s in srcs
            if force or ptxas_verbose
            or _stale(os.path.join(BUILD, os.path.basename(s).replace(".cu", ".o")), [s, *headers])]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4)) as ex:
            for obj, log in ex.map(lambda s: _compile(s, ptxas_verbose), todo):
                if verbose and log.strip():
                    print(f"[{os.path.basename(obj)}]\n{log}", file=sys.stderr)
    objs = [os.path.join(BUILD, os.path.basename(s).replace(".cu", ".o")) for s in srcs]
    if force or todo or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print ptxas resource usage (-Xptxas -v)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose or a.ptxas, ptxas_verbose=a.ptxas))


if __name__ == "__main__":
    main()
