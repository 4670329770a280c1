"""Build libpkv.so (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: python -m paged_kv_sliding_gb300.build [--force] [--verbose]

Each translation unit is compiled in parallel into _build/, then linked into
paged_kv_sliding_gb300/libpkv.so against the shared CUDA runtime.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpkv.so")

SOURCES = ["pkv_api.cpp", "pkv_decode.cu", "pkv_decode_fp8.cu", "pkv_merge.cu", "pkv_prefill.cu",
           "pkv_prefill_fp8.cu",
           "pkv_noalloc.cu", "pkv_indices.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(extra_verbose=False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden", "--use_fast_math",
                "-I", INCLUDE, "-I", CSRC, "-DNDEBUG"]
    f += ["-Xptxas", "-v"]  # the register report is checked (see REGISTER_SPLIT)
    return f


# Kernels that redistribute registers between warpgroups with setmaxnreg: the
# launch allocation (threads x registers per thread) must be exactly what the
# split assumes, or setmaxnreg.inc would wait for registers that never come.
REGISTER_SPLIT = {"pkv_prefill.cu": ("prefill_pp_kernel", 168), "pkv_prefill_fp8.cu": ("prefill_pp_kernel", 168)}


def _check_register_split(logs):
    import re
    for src, (kernel, regs) in REGISTER_SPLIT.items():
        log = logs[src]
        blocks = re.findall(r"Compiling entry function '([^']+)'.*?Used (\d+) registers", log, re.S)
        found = [(name, int(n)) for name, n in blocks if kernel in name]
        if not found:
            raise RuntimeError(f"no ptxas register report for {kernel}")
        bad = [(name, n) for name, n in found if n != regs]
        if bad:
            raise RuntimeError(f"{kernel}: ptxas allocated {bad[0][1]} registers, the register "
                               f"split assumes {regs}")


def _deps_mtime():
    paths = [os.path.join(CSRC, n) for n in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pkv.h")]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime()
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        lang = ["-x", "cu"] if src.endswith(".cu") else []
        cmd = [nvcc] + _flags(verbose) + lang + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    _check_register_split(dict(zip(SOURCES, (log for _, log in results))))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
