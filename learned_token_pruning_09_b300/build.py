"""Build libtokengate.so in-tree with nvcc for sm_103a.

    python -m learned_token_pruning_09_b300.build [--debug]

The library is self-contained (CUDA runtime linked statically; the driver's
cuTensorMapEncodeTiled is resolved at run time), so it loads with or without
PyTorch in the process."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libtokengate.so")
SOURCES = ["tg_api.cu", "tg_gemm.cu", "tg_topk.cu", "tg_gather.cu", "tg_rope.cu", "tg_attention.cu",
           "tg_attention_bwd.cu", "tg_deltanet.cu", "tg_deltanet_chunked.cu", "tg_model.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "tokengate.h"))
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) <= t for d in deps):
            return LIB
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), "-o", LIB + ".tmp", *srcs]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv, force=True)
    print(LIB)
