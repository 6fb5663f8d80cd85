"""fp64 CPU oracle for the ZGCM-1 attention hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library (``global_attention_fwd_b300``) and imports
nothing from it; the product path never calls it.

Two independent CPU implementations live here:

* ``zg_oracle.c`` (built into ``liboracle.so``): the timed, multithreaded
  per-row fp64 oracle for prefill rows and for one decode step of a sequence.
* ``brute.py``: a NumPy full-matrix formulation (explicit L x L mask, RoPE as
  a rotation matrix) for tiny inputs, used to cross-check the C oracle.

Sources (page title, section): "ZGCM-1-7B 完全解説" (gotosocial explainer),
section "アーキテクチャ" (architecture); "ZGCM-1: A Fully Open and Extremely
Efficient Foundation Model for Math and Agentic Search" (jaehun.me review),
section "게이트형 SWA의 동작"; hyper.ai summary of arXiv 2609.13356, section
"方法", GatedSWA equation.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, the pages' printed gate example and KV-cache sizes,
brute force).  The partial-RoPE pairing/frequency convention and the 1/sqrt(d)
softmax scale are fixed by stated reading, not by the pages: parity for those
two choices is unpinned by the pages (both sides share the reading, not code).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

BF16, F64, F32 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile zg_oracle.c with gcc into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", _LIB_PATH, _SRC, "-lm", "-lpthread"]
        subprocess.check_call(cmd)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        I64 = ctypes.c_int64
        lib.zgo_prefill_rows.argtypes = [P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, D, D, P, I64, P, I]
        lib.zgo_prefill_rows.restype = I
        lib.zgo_decode_seq.argtypes = [P, P, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I64, I, I, D, D, I, P, P, I]
        lib.zgo_decode_seq.restype = I
        lib.zgo_rmsnorm.argtypes = [P, P, I, D, P]
        lib.zgo_rmsnorm.restype = None
        lib.zgo_rope.argtypes = [P, I, D, D]
        lib.zgo_rope.restype = None
        lib.zgo_sigmoid.argtypes = [D]
        lib.zgo_sigmoid.restype = D
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _as_input(t):
    """-> (contiguous numpy array holding the data, dtype code)."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy(), BF16
        if t.dtype == torch.float64:
            return t.numpy(), F64
        if t.dtype == torch.float32:
            return t.numpy(), F32
        raise TypeError(f"unsupported dtype {t.dtype}")
    a = np.ascontiguousarray(t)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"unsupported dtype {a.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _f32(t):
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().to(torch.float32).contiguous().numpy()
    return np.ascontiguousarray(t, dtype=np.float32)


def prefill_rows(q, k, v, gate, pos, wq, wk, *, window, rotary_dim, theta, eps, rows, nthreads=None):
    """Attention output of the given query rows, fp64.

    q, gate: [B, L, Hq, d]; k, v: [B, L, Hkv, d] (bf16 / f32 / f64, all the same);
    pos: [B, L] int32; wq, wk: [d].  window <= 0 (or >= L) means full causal
    (the global layer); gate None means ungated.  rows: flattened b*L + i.
    Returns float64 [len(rows), Hq, d].
    """
    lib = _load()
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    qa, dt = _as_input(q)
    ka, dt_k = _as_input(k)
    va, dt_v = _as_input(v)
    ga = None
    if gate is not None:
        ga, dt_g = _as_input(gate)
        assert dt_g == dt
    assert dt == dt_k == dt_v
    pa = np.ascontiguousarray(pos.cpu().numpy() if isinstance(pos, torch.Tensor) else pos, dtype=np.int32)
    wqa, wka = _f32(wq), _f32(wk)
    ra = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(ra), Hq, d), dtype=np.float64)
    rc = lib.zgo_prefill_rows(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), dt, _ptr(pa), _ptr(wqa), _ptr(wka),
                              B, L, Hq, Hkv, d, int(window), int(rotary_dim), float(theta), float(eps),
                              _ptr(ra), len(ra), _ptr(out), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"zgo_prefill_rows failed ({rc})")
    return out


def decode_seq(q, k_new, v_new, gate, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, *,
               p, rotary_dim, theta, eps, nthreads=None):
    """One decode step of ONE sequence through the layer stack, fp64.

    q, gate [NL, Hq, d]; k_new, v_new [NL, Hkv, d]; wq, wk [NL, d];
    is_global [NL] bool; k_glob, v_glob [NG, Hkv, S, d] (this sequence's caches
    as they are before the step); k_ring, v_ring [NS, Hkv, W, d].
    Returns (out [NL, Hq, d], khat_new [NL, Hkv, d]) float64.
    """
    lib = _load()
    NL, Hq, d = q.shape
    Hkv = k_new.shape[1]
    qa, dt = _as_input(q)
    kna, _ = _as_input(k_new)
    vna, _ = _as_input(v_new)
    ga, _ = _as_input(gate)
    wqa, wka = _f32(wq), _f32(wk)
    isg = np.ascontiguousarray(np.asarray(is_global, dtype=np.uint8))
    S = k_glob.shape[2] if k_glob is not None else int(p) + 1
    W = k_ring.shape[2] if k_ring is not None else 1
    cdt = BF16
    kga = vga = kra = vra = None
    if k_glob is not None:
        kga, cdt = _as_input(k_glob)
        vga, _ = _as_input(v_glob)
    if k_ring is not None:
        kra, cdt = _as_input(k_ring)
        vra, _ = _as_input(v_ring)
    out = np.zeros((NL, Hq, d), dtype=np.float64)
    khat = np.zeros((NL, Hkv, d), dtype=np.float64)
    rc = lib.zgo_decode_seq(_ptr(qa), _ptr(kna), _ptr(vna), _ptr(ga), dt, _ptr(wqa), _ptr(wka), _ptr(isg),
                            _ptr(kga), _ptr(vga), _ptr(kra), _ptr(vra), cdt, NL, Hq, Hkv, d, int(S), int(W),
                            int(rotary_dim), float(theta), float(eps), int(p), _ptr(out), _ptr(khat),
                            int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"zgo_decode_seq failed ({rc})")
    return out, khat


def rmsnorm(x, w, eps):
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    y = np.zeros_like(x)
    lib.zgo_rmsnorm(_ptr(x), _ptr(w), x.shape[-1], float(eps), _ptr(y))
    return y


def rope(x, rotary_dim, pos, theta):
    lib = _load()
    y = np.array(x, dtype=np.float64, copy=True)
    lib.zgo_rope(_ptr(y), int(rotary_dim), float(pos), float(theta))
    return y


def sigmoid(x):
    return _load().zgo_sigmoid(float(x))
