"""Builds libpathattn.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into ``_build/`` and then
linked into ``householder_softmax_attention_gb300/libpathattn.so``.  Run
``python -m householder_softmax_attention_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpathattn.so")
SOURCES = ["api.cu", "prep.cu", "prep_tc.cu", "attn_f32.cu", "attn_tc.cu", "bwd.cu", "bwd_tc.cu", "bwd_gemm_tc.cu",
           "decode.cu", "producer.cu", "producer_tc.cu", "producer_mix_tc.cu"]
HEADERS = ["common.cuh", "ptx.cuh", "prep_solve.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(os.path.dirname(HERE), "include", "pathattn.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libpathattn.so."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src + ".log"), "w")
        cmd = [cc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    failed = []
    for src, p, log in procs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src + ".log")) as f:
                msgs.append(f"--- {src}\n" + f.read()[-4000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    if verbose:
        for src in SOURCES:
            with open(os.path.join(BUILD, src + ".log")) as f:
                sys.stdout.write(f.read())
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart=static"],
                   check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
