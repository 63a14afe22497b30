"""Build libbitdelta.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file,
then nvcc links them into ``bit_delta_tenant_gb300/lib/libbitdelta.so`` with
the CUDA runtime linked statically and only the ``bd_*`` symbols exported.
Re-running is cheap: a unit is rebuilt only when it or a header is newer than
its object.  ``debug=True`` builds the bounds-checked variant (``-DBD_DEBUG``:
kernels check their global indices and record failures in the device status
word) into ``lib/libbitdelta_debug.so`` from objects of its own.
Usage: ``python -m bit_delta_tenant_gb300.build [--force] [-v] [--debug]``.
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
LIB_DIR = os.path.join(PKG, "lib")


def _paths(debug: bool):
    """(object directory, library path) of the release or the bounds-checked build."""
    if debug:
        return os.path.join(PKG, "_build_debug"), os.path.join(LIB_DIR, "libbitdelta_debug.so")
    return os.path.join(PKG, "_build"), os.path.join(LIB_DIR, "libbitdelta.so")


OBJ_DIR, LIB_PATH = _paths(False)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbitdelta.so")
    return exe


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src: str, force: bool, verbose: bool, ptxas_info: bool, obj_dir: str, debug: bool) -> str:
    obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
    if (not force and os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
            and os.path.getmtime(obj) >= _headers_mtime()):
        return obj
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DBD_DEBUG"] if debug else []), "-c", src, "-o", obj + ".tmp"]
    if ptxas_info:
        cmd.insert(1, "-Xptxas=-v")
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    if ptxas_info or verbose:
        sys.stdout.write(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    obj_dir, lib_path = _paths(debug)
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, force, verbose, ptxas_info, obj_dir, debug), sources))
    newest = max(os.path.getmtime(o) for o in objs)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest:
        return lib_path
    vscript = os.path.join(obj_dir, "exports.map")
    with open(vscript, "w") as f:
        f.write("{ global: bd_*; local: *; };\n")
    tmp = lib_path + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart=static", "-Xcompiler", "-fPIC",
           f"-Xlinker=--version-script={vscript}", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the bounds-checked build (libbitdelta_debug.so)")
    args = ap.parse_args()
    print(build(args.force, args.verbose, args.ptxas_info, args.debug))
