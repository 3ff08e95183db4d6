"""Builds libtq_gb300.so in-tree with nvcc for sm_103a (GB300).

Usage: ``python -m quantized_kv_cache_06_gb300.build`` or ``build_library()``.
Translation units compile in parallel; the shared library links the CUDA runtime
statically so that it does not depend on the loader finding libcudart.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libtq_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["tq_api.cpp", "tq_write.cu", "tq_write_tc.cu", "tq_decode.cu", "tq_decode_tc.cu", "tq_decode_tc_a.cu",
           "tq_decode_tc_b.cu", "tq_decode_tc_c.cu", "tq_decode_tc_d.cu", "tq_decode_tc_e.cu",
           "tq_decode_tc_f.cu", "tq_decode_tc_p.cu",
           "tq_decode_tc_q.cu", "tq_prefill_mq.cu",
           "tq_dequant.cu", "tq_qjl.cu", "tq_recipe.cu", "tq_query.cu",
           "tq_small.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the TurboQuant GB300 library needs the CUDA 13 toolkit")
    return cand


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc_path(), "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *ARCH, *extra]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip():
        sys.stderr.write(res.stderr)
    return obj


def build_library(verbose_ptxas: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "tq.h"))
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(p) for p in deps)
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc_path(), "-shared", "-o", tmp, *objs, *ARCH, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(verbose_ptxas="-v" in sys.argv, force="-f" in sys.argv))
