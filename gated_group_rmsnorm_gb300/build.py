"""Build ``libggrn.so`` (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file.  ``python -m gated_group_rmsnorm_gb300.build``
runs it; ``--ptxas-v`` also prints the register/shared-memory usage that ptxas
reports for every kernel.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(HERE, "libggrn.so")
BUILD_DIR = os.path.join(HERE, "_build")
# profiling build: the same library with the streaming kernels' per-CTA
# timeline compiled in (-DGGRN_TIMELINE); never loaded by the product path
TIMELINE_LIB_PATH = os.path.join(HERE, "libggrn_timeline.so")
TIMELINE_BUILD_DIR = os.path.join(HERE, "_build_timeline")

SOURCES = ["ggrn_api.cu", "ggrn_host.cu", "ggrn_kernels_bf16.cu", "ggrn_kernels_f16.cu",
           "ggrn_kernels_f32.cu", "ggrn_outproj.cu"]
HEADERS = ["ggrn_internal.h", "ggrn_kernels.cuh", "ggrn_slots.h", "ggrn_stream.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libggrn.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _deps() -> list[str]:
    return ([os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in HEADERS] +
            [os.path.join(INCLUDE, "ggrn.h"), os.path.abspath(__file__)])


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True,
          timeline: bool = False) -> str:
    """Compile and link ``libggrn.so`` (``timeline``: the profiling build
    ``libggrn_timeline.so``); return its path.  No-op when up to date."""
    lib_path = TIMELINE_LIB_PATH if timeline else LIB_PATH
    build_dir = TIMELINE_BUILD_DIR if timeline else BUILD_DIR
    if not force and not ptxas_verbose and not _stale(lib_path, _deps()):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if timeline:
        extra += ["-DGGRN_TIMELINE"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", os.path.join(CSRC, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if ptxas_verbose or not quiet:
        for _, log in results:
            sys.stdout.write(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true")
    ap.add_argument("--timeline", action="store_true",
                    help="the profiling build with the per-CTA timeline (libggrn_timeline.so)")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.ptxas_v, quiet=False,
                timeline=args.timeline))
