"""Builds libmdcn.so in-tree with nvcc for sm_103a (no cmake).

    python -m modulated_deformable_convolution_gb300.build [--force]

Objects go to ``_build/`` beside this file; translation units compile in
parallel; ptxas resource usage (registers, shared memory, spills) is written
to ``_build/ptxas.log``.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmdcn.so")

CU_SOURCES = ["mdcn_fused.cu", "mdcn_prep.cu", "mdcn_im2col.cu", "mdcn_noalloc.cu", "mdcn_backward.cu", "mdcn_gemm.cu",
              "mdcn_direct.cu"]
CPP_SOURCES = ["mdcn_api.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def _headers():
    out = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh")):
                out.append(os.path.join(d, f))
    return out


def _stale(obj: str, src: str, headers) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src, *headers, __file__])


def _compile(cmd, log_path=None):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if log_path is not None:
        with open(log_path, "w") as f:
            f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("compile failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    headers = _headers()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC"]
    jobs = []
    objs = []
    for src in CU_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or _stale(o, s, headers):
            cmd = [nvcc, *ARCH, "-lineinfo", "-Xptxas", "-v", *common, "-c", s, "-o", o]
            jobs.append((cmd, os.path.join(BUILD, src + ".ptxas.log")))
    for src in CPP_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or _stale(o, s, headers):
            cmd = [nvcc, *ARCH, *common, "-x", "c++", "-c", s, "-o", o]
            jobs.append((cmd, None))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            futs = [ex.submit(_compile, c, l) for c, l in jobs]
            for f in futs:
                out = f.result()
                if verbose and out:
                    print(out)
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            for src in CU_SOURCES:
                p = os.path.join(BUILD, src + ".ptxas.log")
                if os.path.exists(p):
                    f.write(open(p).read())
    if force or jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        lib64 = os.path.join(home, "lib64")
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcublas", "-Xlinker", f"-rpath,{lib64}"]
        _compile(cmd)
        os.replace(tmp, LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    sys.exit(main())
