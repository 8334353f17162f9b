"""Builds libdsa_gb300.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

The translation units compile in parallel; the result sits next to this file, where
the ctypes binding loads it.  Usage: ``python -m deepseek_v4_sparse_dsa_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdsa_gb300.so")

SOURCES = ["indexer_bf16_topk.cu", "indexer_fp8_topk.cu", "indexer_bf16_logits.cu", "indexer_fp8_logits.cu",
           "api.cu", "gather.cu", "indexer.cu", "topk.cu", "noalloc.cu", "producer.cu",
           "sparse_attn.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(src: str, nvcc: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(BUILD, src + ".log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    return obj


def build(verbose: bool = False, extra=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc, list(extra)), SOURCES))
    tmp = LIB + ".tmp"
    # The CUDA runtime is linked statically; the driver entry point used for tensor
    # maps is looked up through it, so the library loads on hosts without a driver.
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        for s in SOURCES:
            with open(os.path.join(BUILD, s + ".log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
