"""Builds libmoe_lora.so, the C-ABI library, in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the shared object lands next to
this file and the objects under ``_build/``. Run ``python -m
expert_adapter_gemms_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libmoe_lora.so")
SOURCES = ["route.cu", "align.cu", "grouped_gemm.cu", "fused_gemm.cu", "lora_shrink.cu",
           "lora_expand.cu", "layer.cu", "layer_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "-Xcompiler", "-Wall",
                   "-I", os.path.join(HERE, "..", "include")] + list(extra)


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + p.stdout)
    return p.stdout


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compiles every CUDA source and links the shared library; returns its path."""
    home = _cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(HERE, "..", "include", "moe_lora.h"))
    newest_header = max(os.path.getmtime(h) for h in headers)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        if (not force and not ptxas_info and os.path.exists(o)
                and os.path.getmtime(o) >= max(os.path.getmtime(s), newest_header)):
            return o, ""
        out = _run([nvcc] + _flags(extra) + ["-c", s, "-o", o])
        return o, out

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(one, SOURCES))
    objs = [o for o, _ in results]
    if verbose or ptxas_info:
        for (o, out) in results:
            if out:
                sys.stdout.write(f"== {os.path.basename(o)}\n{out}")
    tmp = LIB_PATH + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs +
         ["-Xlinker", "-rpath=" + os.path.join(home, "lib64")])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv))
