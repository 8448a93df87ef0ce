"""Builds libmoe.so in-tree for sm_103a: one nvcc per translation unit, in parallel, then link.

    python -m routing_expert_ffn_gb300.build [--verbose-ptxas]

Objects go to routing_expert_ffn_gb300/_build/, the library to
routing_expert_ffn_gb300/libmoe.so.  A translation unit is recompiled when it
or any header under csrc/ or include/ is newer than its object.

build(fault=True) builds the fault-injection test variant instead: the same sources with
-DMOE_FAULT_INJECTION (bounded waits give up after 50 ms, and moe_test_drop_gemm_loads
makes the GEMM's loads never arrive), into _build_fault/ and libmoe_fault.so.  Only the
timeout test loads it.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")
BUILD_FAULT = os.path.join(PKG, "_build_fault")
LIB_FAULT = os.path.join(PKG, "libmoe_fault.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(verbose_ptxas: bool = False, force: bool = False, fault: bool = False) -> str:
    BUILD = BUILD_FAULT if fault else globals()["BUILD"]
    LIB = LIB_FAULT if fault else globals()["LIB"]
    extra = ["-DMOE_FAULT_INJECTION"] if fault else []
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _headers_mtime()
    cc = nvcc()

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
                and os.path.getmtime(obj) >= hdr_t and not verbose_ptxas):
            return obj, ""
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose_ptxas:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose_ptxas:
        for obj, log in results:
            sys.stderr.write(f"== {os.path.basename(obj)}\n{log}")
    objs = [o for o, _ in results]
    if force or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        cmd = [cc, *ARCH, "-shared", "-o", LIB, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--fault", action="store_true", help="the fault-injection test variant")
    a = ap.parse_args()
    print(build(a.verbose_ptxas, a.force, a.fault))
