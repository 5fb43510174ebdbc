"""Build libda.so, the sm_103a deformable-aggregation library, in-tree.

Every .cu file under csrc/ is compiled to its own object in parallel, and the
objects are linked into deformable_view_feature_gb300/_build/libda.so. The
CUDA runtime is linked statically. nvcc cross-compiles, so this needs no GPU.

--debug-bounds builds the bounds-checking variant instead
(_build/debug/libda_debug.so, compiled with DA_DEBUG_BOUNDS): every index a
kernel computes is checked before use, and the entry points return
DA_ERR_DEVICE_BOUNDS when one was outside its tensor (include/da.h). The
binding loads it when the environment variable DA_DEBUG_BOUNDS is 1.

    python -m deformable_view_feature_gb300.build [--force] [--verbose] [--debug-bounds]
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libda.so")
DEBUG_DIR = os.path.join(OUT_DIR, "debug")
DEBUG_LIB = os.path.join(DEBUG_DIR, "libda_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libda.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool | None = None) -> str:
    """Compile and link libda.so (libda_debug.so with debug_bounds) unless it
    is newer than every source; return its path. debug_bounds=None follows
    the environment variable DA_DEBUG_BOUNDS, as the binding's loader does."""
    if debug_bounds is None:
        debug_bounds = os.environ.get("DA_DEBUG_BOUNDS") == "1"
    out_dir, lib = (DEBUG_DIR, DEBUG_LIB) if debug_bounds else (OUT_DIR, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    srcs = _sources()
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = ["-Xptxas", "-v"] if verbose else []
    if debug_bounds:
        extra += ["-DDA_DEBUG_BOUNDS=1"]

    def compile_one(pair):
        src, obj = pair
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    for src, r in results:
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="pass -Xptxas -v and print its report")
    ap.add_argument("--debug-bounds", action="store_true", default=None,
                    help="build the bounds-checking libda_debug.so")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, debug_bounds=a.debug_bounds))
