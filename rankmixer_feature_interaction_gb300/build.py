"""Build librankmixer.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into rankmixer_feature_interaction_gb300/librankmixer.so
with the CUDA runtime linked statically.  Rebuilds only what changed.

--debug-bounds builds the bounds-checked variant instead (-DRM_DEBUG_BOUNDS:
launcher checks of sizes, strides and alignments, and device-side guards that
latch an error word and skip the access), as librankmixer_debug.so; the
binding loads it when RM_LIBRARY=debug is set.

    python -m rankmixer_feature_interaction_gb300.build [--force] [--debug-bounds] [-v]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build", "rankmixer")
LIB_PATH = os.path.join(PKG_DIR, "librankmixer.so")
DEBUG_BUILD_DIR = os.path.join(ROOT, "_build", "rankmixer_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "librankmixer_debug.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build librankmixer.so)")


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src: str, obj: str, verbose: bool, extra: list[str]) -> str:
    cmd = [nvcc_path()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout.strip() or r.stderr.strip()):
        print(r.stdout + r.stderr, flush=True)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug_bounds: bool = False) -> str:
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _headers_mtime()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if debug_bounds:
        extra = extra + ["-DRM_DEBUG_BOUNDS"]
    jobs = []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        if force or ptxas_verbose or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), hdr_t):
            jobs.append((s, o))
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = [ex.submit(_compile, s, o, verbose or ptxas_verbose, extra) for s, o in jobs]
            for f in futs:
                f.result()
    need_link = force or bool(jobs) or not os.path.exists(lib_path) or \
        os.path.getmtime(lib_path) < max(os.path.getmtime(o) for o in objs)
    if need_link:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc_path()] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs + ["-Xcompiler", "-fPIC"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true", help="print registers/spills/smem per kernel")
    ap.add_argument("--debug-bounds", action="store_true",
                    help="build the bounds-checked variant librankmixer_debug.so (-DRM_DEBUG_BOUNDS)")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose, debug_bounds=a.debug_bounds))
    return 0


if __name__ == "__main__":
    sys.exit(main())
