"""Builds libtkg.so in-tree: each CUDA translation unit compiled for sm_103a
in parallel with nvcc, then linked into one shared library.  With --check it
builds libtkg_check.so instead: the same sources with TKG_CHECK=1, every
kernel verifying its internal invariants (include/tkg_gemm.h, check builds).

    python -m dense_block_scaled_gb300.build [--force] [--verbose] [--check]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtkg.so")
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "libtkg_check.so")
SOURCES = ["tkg_api.cu", "quantize.cu", "gemm_bf16.cu", "gemm_mxfp8.cu", "gemm_nvfp4.cu", "gemm_noalloc.cu",
           "gemm_grouped.cu", "host_pipeline.cu", "gemm_list.cu"]
HEADERS = ["ptx.cuh", "gemm_kernel.cuh", "gemm_splitk.cuh", "host_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    build_dir, lib_path = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DTKG_CHECK=1"] if check else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "tkg_gemm.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [nvcc, *ARCH, *flags, "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for s, r in ex.map(compile_one, jobs):
                if verbose or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {os.path.basename(s)}")
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".{os.getpid()}.tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"link of {os.path.basename(lib_path)} failed")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--check", action="store_true", help="build libtkg_check.so (kernels verify their invariants)")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, check=a.check))
