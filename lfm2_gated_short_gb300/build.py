"""Build libshortconv.so in-tree for sm_103a.

Compiles every ``csrc/*.cu`` translation unit with nvcc in parallel and links
them into ``lfm2_gated_short_gb300/_build/libshortconv.so`` (CUDA runtime
linked statically, so the library needs only the driver at run time).

``--bounds-check`` builds the same sources with ``-DSC_BOUNDS_CHECK`` into
``_build/bounds/libshortconv.so``: every global access the kernels make
through their memory helpers is checked against the buffers of the call
(see shortconv_bounds_checked in include/shortconv.h). It is for tests.

    python -m lfm2_gated_short_gb300.build [--force] [--ptxas-verbose] [--bounds-check]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libshortconv.so")
BOUNDS_DIR = os.path.join(BUILD_DIR, "bounds")
BOUNDS_LIB_PATH = os.path.join(BOUNDS_DIR, "libshortconv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libshortconv.so")
    return cand


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True,
          bounds_check: bool = False) -> str:
    """Compile and link; return the library path. Skips work when up to date."""
    out_dir = BOUNDS_DIR if bounds_check else BUILD_DIR
    lib_path = BOUNDS_LIB_PATH if bounds_check else LIB_PATH
    if not force and not ptxas_verbose and not is_stale(lib_path):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if bounds_check:
        extra.append("-DSC_BOUNDS_CHECK")

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if (ptxas_verbose or not quiet) and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_all() -> None:
    """The standard library and the bounds-checked one, side by side."""
    with cf.ThreadPoolExecutor(2) as ex:
        for f in [ex.submit(build), ex.submit(build, bounds_check=True)]:
            f.result()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--bounds-check", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False,
                bounds_check=a.bounds_check))


if __name__ == "__main__":
    main()
