"""Build libzgattn.so in-tree with nvcc for sm_103a (no JIT cache, no torch extension).

Each source is compiled to an object in parallel, then linked.  `build(debug=True)` makes
libzgattn_debug.so instead: the same kernels compiled with ZG_DEBUG, whose plain global-memory
indices are checked before every access (a bad one is recorded in the device error word and
the access skipped)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libzgattn.so")
LIB_DEBUG = os.path.join(HERE, "libzgattn_debug.so")
OBJ_DIR = os.path.join(HERE, "..", "_build")
SOURCES = ["api.cu", "swa_prefill.cu", "swa2_prefill.cu", "global_prefill.cu", "hybrid_decode.cu", "selftest.cu",
           "noalloc.cu", "kv_cache.cu", "attn_backward.cu", "attn_backward_tc.cu", "gemm.cu"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]
LDFLAGS = ["-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64"]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "zg_attn.h")]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    tag = "debug" if debug else "release"
    odir = os.path.join(OBJ_DIR, tag)
    os.makedirs(odir, exist_ok=True)
    extra = (["-DZG_DEBUG"] if debug else []) + (["-Xptxas", "-v"] if verbose else [])
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]

    def compile_one(s):
        obj = os.path.join(odir, s.replace(".cu", ".o"))
        subprocess.check_call([NVCC, *ARCH, *CFLAGS, *extra, "-c", "-o", obj, os.path.join(CSRC, s)])
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, srcs))
    subprocess.check_call([NVCC, *ARCH, *LDFLAGS, "-o", lib + ".tmp", *objs])
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
