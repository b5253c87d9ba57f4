"""Build libfa.so (the CUDA library behind include/fa.h) in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into
``libfa.so`` beside this file.  Only a GB300-class toolchain target is
built: ``-gencode arch=compute_103a,code=sm_103a``.  The kernel variants of
``ablate_*.cu`` make ``libfa_ablate.so`` (include/fa_ablate.h), linked
against libfa.so; only the benchmark's ablation mode and its test load it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa.so")
LIB_ABLATE = os.path.join(HERE, "libfa_ablate.so")
UNITS = ["api.cu", "attn_bf16.cu", "attn_fp16.cu", "attn_fp8.cu", "quant_fp8.cu", "quant_fp8_noalloc.cu",
         "splitkv.cu", "attn_split_bf16.cu", "attn_split_fp16.cu", "attn_bwd.cu"]
ABLATE_UNITS = ["ablate_api.cu", "ablate_bf16.cu", "ablate_bf16_causal.cu", "ablate_fp8.cu", "ablate_d64.cu"]
HEADERS = ["ptx.cuh", "attn_fwd.cuh", "quant_fp8.h", "attn_bwd.h", "splitkv.h", "ablate_inst.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", INCLUDE,
                   "--expt-relaxed-constexpr"] + list(extra)


def _stale(out, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, h) for h in ("fa.h", "fa_ablate.h")]
    objs = []
    ablate_objs = []
    jobs = []
    for u in UNITS + ABLATE_UNITS:
        src = os.path.join(CSRC, u)
        obj = os.path.join(BUILD, u.replace(".cu", ".o"))
        (objs if u in UNITS else ablate_objs).append(obj)
        if force or _stale(obj, [src] + hdrs):
            jobs.append([nvcc()] + _flags(extra_flags) + ["-c", src, "-o", obj])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    # the ablation library holds only its kernel variants and links against
    # libfa.so (found beside it), so no kernel is loaded twice in a process
    for lib, lobjs, extra in ((LIB, objs, []),
                              (LIB_ABLATE, ablate_objs, ["-L" + HERE, "-lfa", "-Xlinker", "-rpath,$ORIGIN"])):
        if force or jobs or _stale(lib, lobjs + ([LIB] if extra else [])):
            cmd = [nvcc()] + ARCH + ["-shared", "-o", lib + ".tmp"] + lobjs + extra
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
                raise RuntimeError(f"link of {os.path.basename(lib)} failed")
            os.replace(lib + ".tmp", lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
