"""Build the MIS shared library for sm_103a with nvcc (no cmake).

Produces ``ranking_prefill_gb300/libmis_gb300.so`` in-tree. Object files go
to ``ranking_prefill_gb300/_build/``. Translation units compile in parallel.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmis_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CU_SOURCES = ["mis_attn.cu", "mis_score.cu", "mis_rope.cu"]
CPP_SOURCES = ["mis_plan.cpp", "mis_abi.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I", CSRC]
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        flags = ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]
        if ptxas_info:
            flags += ["-Xptxas", "-v"]
        jobs.append([nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common + flags)
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append([nvcc, "-c", "-x", "c++", os.path.join(CSRC, src), "-o", obj] + common)
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(_run, jobs))
    objs = [os.path.join(BUILD, s + ".o") for s in CU_SOURCES + CPP_SOURCES]
    tmp = LIB + ".tmp"
    logs.append(_run([nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]))
    os.replace(tmp, LIB)
    out = "\n".join(l for l in logs if l.strip())
    if verbose and out:
        print(out, file=sys.stderr)
    return out


if __name__ == "__main__":
    print(build(verbose=False, ptxas_info="-v" in sys.argv) or "built " + LIB)
