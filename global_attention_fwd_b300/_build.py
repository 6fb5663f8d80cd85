"""Build libzgattn.so in-tree with nvcc for sm_103a (no JIT cache, no torch extension)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libzgattn.so")
SOURCES = ["api.cu", "swa_prefill.cu", "swa2_prefill.cu", "global_prefill.cu", "hybrid_decode.cu", "selftest.cu", "noalloc.cu", "kv_cache.cu", "layer.cu", "attn_backward.cu", "attn_backward_tc.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-shared",
    "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
    "--expt-relaxed-constexpr",
    "-lcublasLt",
]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "zg_attn.h")]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    srcs = [os.path.join(CSRC, s) for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    cmd = [NVCC, *FLAGS, *( ["-Xptxas", "-v"] if verbose else []), "-o", LIB + ".tmp", *srcs]
    subprocess.check_call(cmd)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
