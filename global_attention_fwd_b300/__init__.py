"""Python binding of libzgattn.so, the ZGCM-1 attention hot path for B300.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, and their pointers and the current CUDA stream are passed to the
C ABI declared in ``include/zg_attn.h``.  Every step of the computation runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
importing this package fails if the library cannot be loaded.

Entry points (same names as the C ABI without the ``zg_`` prefix):
``swa_prefill``, ``global_prefill``, ``global_prefill_workspace_bytes``,
``hybrid_decode``, ``hybrid_decode_workspace_bytes``, ``device_status``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ZG_LIBRARY=debug selects libzgattn_debug.so, the same kernels with device-side index checks
LIB_PATH = os.path.join(_HERE, "libzgattn_debug.so" if os.environ.get("ZG_LIBRARY") == "debug" else "libzgattn.so")

STATUS = {
    0: "ZG_OK", -1: "ZG_ERR_NULL", -2: "ZG_ERR_ALIGN", -3: "ZG_ERR_SHAPE", -4: "ZG_ERR_UNSUPPORTED",
    -5: "ZG_ERR_POSITION", -6: "ZG_ERR_WORKSPACE", -7: "ZG_ERR_CUDA", -8: "ZG_ERR_DEVICE_TIMEOUT",
    -9: "ZG_ERR_UNIMPLEMENTED", -10: "ZG_ERR_DEVICE_INDEX",
}
EXPORTS = ("zg_swa_prefill", "zg_swa_prefill_host_workspace_bytes", "zg_swa_prefill_host", "zg_global_prefill_workspace_bytes", "zg_global_prefill",
           "zg_swa_prefill_with_cache", "zg_global_prefill_with_cache", "zg_kv_cache_write",
           "zg_gated_swa_layer_workspace_bytes", "zg_gated_swa_layer", "zg_linear",
           "zg_attention_backward_workspace_bytes", "zg_attention_backward",
           "zg_hybrid_decode_workspace_bytes", "zg_hybrid_decode", "zg_hybrid_decode_noalloc",
           "zg_hybrid_decode_fp8", "zg_kv_cache_write_fp8", "zg_global_prefill_fp8_workspace_bytes",
           "zg_global_prefill_fp8", "zg_swa_prefill_fp8",
           "zg_device_status", "zg_selftest_bounded_wait", "zg_selftest_index_check", "zg_debug_build",
           "zg_status_string")


class ZgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_lib.zg_status_string(status).decode()})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m global_attention_fwd_b300._build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, D, F, SZ, U64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float,
                                ctypes.c_size_t, ctypes.c_uint64)
    lib.zg_swa_prefill.argtypes = [P] * 8 + [I] * 7 + [D, F, P]
    lib.zg_swa_prefill.restype = I
    lib.zg_swa_prefill_host_workspace_bytes.argtypes = [I] * 6
    lib.zg_swa_prefill_host_workspace_bytes.restype = SZ
    lib.zg_swa_prefill_host.argtypes = [P] * 8 + [I] * 7 + [D, F, I, P, SZ, P]
    lib.zg_swa_prefill_host.restype = I
    lib.zg_global_prefill_workspace_bytes.argtypes = [I, I, I, I]
    lib.zg_global_prefill_workspace_bytes.restype = SZ
    lib.zg_global_prefill.argtypes = [P] * 7 + [I] * 6 + [D, F, P, SZ, P]
    lib.zg_global_prefill.restype = I
    lib.zg_swa_prefill_with_cache.argtypes = [P] * 8 + [I] * 7 + [D, F, P, P, I, P]
    lib.zg_swa_prefill_with_cache.restype = I
    lib.zg_global_prefill_with_cache.argtypes = [P] * 7 + [I] * 6 + [D, F, P, SZ, P, P, I64, P]
    lib.zg_global_prefill_with_cache.restype = I
    lib.zg_kv_cache_write.argtypes = [P] * 6 + [I] * 4 + [I64, I, I, D, F, P]
    lib.zg_kv_cache_write.restype = I
    lib.zg_gated_swa_layer_workspace_bytes.argtypes = [I] * 5
    lib.zg_gated_swa_layer_workspace_bytes.restype = SZ
    lib.zg_gated_swa_layer.argtypes = [P] * 10 + [I] * 8 + [D, F, P, SZ, P]
    lib.zg_gated_swa_layer.restype = I
    lib.zg_linear.argtypes = [P, P, P, I64, I, I, P]
    lib.zg_linear.restype = I
    lib.zg_attention_backward_workspace_bytes.argtypes = [I] * 5
    lib.zg_attention_backward_workspace_bytes.restype = SZ
    lib.zg_attention_backward.argtypes = [P] * 12 + [I] * 7 + [D, F, P, SZ, P]
    lib.zg_attention_backward.restype = I
    lib.zg_hybrid_decode_workspace_bytes.argtypes = [I, I, I, I, I64]
    lib.zg_hybrid_decode_workspace_bytes.restype = SZ
    lib.zg_hybrid_decode.argtypes = [P] * 13 + [I] * 5 + [I64, I, I, D, F, P, SZ, P]
    lib.zg_hybrid_decode.restype = I
    lib.zg_hybrid_decode_fp8.argtypes = [P] * 13 + [I] * 5 + [I64, I, I, D, F, F, F, P, SZ, P]
    lib.zg_hybrid_decode_fp8.restype = I
    lib.zg_kv_cache_write_fp8.argtypes = [P] * 6 + [I] * 4 + [I64, I, I, D, F, F, F, P]
    lib.zg_kv_cache_write_fp8.restype = I
    lib.zg_global_prefill_fp8_workspace_bytes.argtypes = [I, I, I, I]
    lib.zg_global_prefill_fp8_workspace_bytes.restype = SZ
    lib.zg_global_prefill_fp8.argtypes = [P] * 7 + [I] * 6 + [D, F, F, F, F, P, SZ, P]
    lib.zg_global_prefill_fp8.restype = I
    lib.zg_swa_prefill_fp8.argtypes = [P] * 8 + [I] * 7 + [D, F, F, F, F, P, SZ, P]
    lib.zg_swa_prefill_fp8.restype = I
    lib.zg_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.zg_device_status.restype = I
    lib.zg_selftest_bounded_wait.argtypes = [U64, P]
    lib.zg_selftest_bounded_wait.restype = I
    lib.zg_selftest_index_check.argtypes = [P]
    lib.zg_selftest_index_check.restype = I
    lib.zg_debug_build.argtypes = []
    lib.zg_debug_build.restype = I
    lib.zg_status_string.argtypes = [I]
    lib.zg_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()
lib = _lib  # raw ctypes handle: the C ABI itself


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, dtype, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _raise(st, what):
    if st != 0:
        raise ZgError(st, what)


def swa_prefill(q, k, v, gate, pos, wq, wk, *, window=128, rotary_dim, theta, eps=1e-6, out=None, stream=None):
    """Gated sliding-window GQA prefill.  q, gate [B,L,Hq,d] bf16; k, v [B,L,Hkv,d] bf16;
    pos [B,L] int32; wq, wk [d] float32.  Returns out [B,L,Hq,d] bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate, "gate")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 4)
    st = _lib.zg_swa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                             B, L, Hq, Hkv, d, int(window), int(rotary_dim), float(theta), float(eps), _stream(stream))
    _raise(st, "zg_swa_prefill")
    return out


def swa_prefill_host_workspace_bytes(B, Hq, Hkv, d, window=128, chunk_tokens=16384) -> int:
    return int(_lib.zg_swa_prefill_host_workspace_bytes(int(B), int(Hq), int(Hkv), int(d), int(window),
                                                        int(chunk_tokens)))


def _check_host(t, name, dtype, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def swa_prefill_host(q, k, v, gate, pos, wq, wk, *, window=128, rotary_dim, theta, eps=1e-6, out=None,
                     chunk_tokens=16384, workspace=None, stream=None):
    """swa_prefill on HOST tensors (pinned for overlap): the copies to and from the device happen inside the
    call, chunk by chunk, overlapped with the kernel.  workspace: optional uint8 CUDA tensor of
    >= swa_prefill_host_workspace_bytes() bytes.  Returns out (host, bf16)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate, "gate")):
        _check_host(t, n, torch.bfloat16, 4)
    _check_host(pos, "pos", torch.int32, 2)
    _check_host(wq, "wq", torch.float32)
    _check_host(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty(B, L, Hq, d, dtype=torch.bfloat16, pin_memory=True)
    _check_host(out, "out", torch.bfloat16, 4)
    need = swa_prefill_host_workspace_bytes(B, Hq, Hkv, d, window, chunk_tokens)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_swa_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                                  B, L, Hq, Hkv, d, int(window), int(rotary_dim), float(theta), float(eps),
                                  int(chunk_tokens), _ptr(workspace), ws_bytes, _stream(stream))
    _raise(st, "zg_swa_prefill_host")
    return out


def global_prefill_workspace_bytes(B, L, Hkv, d) -> int:
    return int(_lib.zg_global_prefill_workspace_bytes(int(B), int(L), int(Hkv), int(d)))


def global_prefill(q, k, v, pos, wq, wk, *, rotary_dim, theta, eps=1e-6, out=None, workspace=None, stream=None):
    """Global (full causal, ungated) GQA prefill.  Same layouts as swa_prefill without gate.
    workspace: optional uint8 CUDA tensor of >= global_prefill_workspace_bytes() bytes."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 4)
    need = global_prefill_workspace_bytes(B, L, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_global_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                                B, L, Hq, Hkv, d, int(rotary_dim), float(theta), float(eps), _ptr(workspace),
                                ws_bytes, _stream(stream))
    _raise(st, "zg_global_prefill")
    return out


def global_prefill_fp8_workspace_bytes(B, L, Hkv, d) -> int:
    return int(_lib.zg_global_prefill_fp8_workspace_bytes(int(B), int(L), int(Hkv), int(d)))


def global_prefill_fp8(q, k, v, pos, wq, wk, *, q_scale=1.0, k_scale=1.0, v_scale=1.0, rotary_dim, theta, eps=1e-6,
                       out=None, workspace=None, stream=None):
    """global_prefill on E4M3 inputs: q [B,L,Hq,d], k, v [B,L,Hkv,d] uint8 holding e4m3(x * scale);
    products on the E4M3 tensor-core path.  Returns out [B,L,Hq,d] bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.uint8, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty(B, L, Hq, d, dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, 4)
    need = global_prefill_fp8_workspace_bytes(B, L, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_global_prefill_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                                    B, L, Hq, Hkv, d, int(rotary_dim), float(theta), float(eps), float(q_scale),
                                    float(k_scale), float(v_scale), _ptr(workspace), ws_bytes, _stream(stream))
    _raise(st, "zg_global_prefill_fp8")
    return out


def swa_prefill_fp8(q, k, v, gate, pos, wq, wk, *, window=128, q_scale=1.0, k_scale=1.0, v_scale=1.0, rotary_dim,
                    theta, eps=1e-6, out=None, workspace=None, stream=None):
    """swa_prefill on E4M3 inputs: q [B,L,Hq,d], k, v [B,L,Hkv,d] uint8 holding e4m3(x * scale); gate
    [B,L,Hq,d] bf16.  Products on the E4M3 tensor-core path.  Returns out [B,L,Hq,d] bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.uint8, 4)
    _check(gate, "gate", torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty(B, L, Hq, d, dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16, 4)
    need = global_prefill_fp8_workspace_bytes(B, L, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_swa_prefill_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                                 B, L, Hq, Hkv, d, int(window), int(rotary_dim), float(theta), float(eps),
                                 float(q_scale), float(k_scale), float(v_scale), _ptr(workspace), ws_bytes,
                                 _stream(stream))
    _raise(st, "zg_swa_prefill_fp8")
    return out


def swa_prefill_with_cache(q, k, v, gate, pos, wq, wk, k_ring, v_ring, *, window=128, rotary_dim, theta, eps=1e-6,
                           out=None, stream=None):
    """swa_prefill, then this local layer's decode rings: k_ring, v_ring [B,Hkv,W,d] bf16 receive
    k_hat and v of the last min(L, W) tokens at slot pos mod W (W = k_ring.shape[2])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (gate, "gate"), (k_ring, "k_ring"), (v_ring, "v_ring")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 4)
    st = _lib.zg_swa_prefill_with_cache(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk),
                                        _ptr(out), B, L, Hq, Hkv, d, int(window), int(rotary_dim), float(theta),
                                        float(eps), _ptr(k_ring), _ptr(v_ring), int(k_ring.shape[2]), _stream(stream))
    _raise(st, "zg_swa_prefill_with_cache")
    return out


def global_prefill_with_cache(q, k, v, pos, wq, wk, k_cache, v_cache, *, rotary_dim, theta, eps=1e-6, out=None,
                              workspace=None, stream=None):
    """global_prefill, then this global layer's decode caches: k_cache, v_cache [B,Hkv,S_max,d] bf16
    receive k_hat and v of every token at slot pos (S_max = k_cache.shape[2])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 4)
    need = global_prefill_workspace_bytes(B, L, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_global_prefill_with_cache(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(out),
                                           B, L, Hq, Hkv, d, int(rotary_dim), float(theta), float(eps),
                                           _ptr(workspace), ws_bytes, _ptr(k_cache), _ptr(v_cache),
                                           int(k_cache.shape[2]), _stream(stream))
    _raise(st, "zg_global_prefill_with_cache")
    return out


def kv_cache_write(k, v, pos, wk, k_cache, v_cache, *, ring, rotary_dim, theta, eps=1e-6, stream=None):
    """Decode caches from prefill keys / values: k_cache, v_cache [B,Hkv,S,d] bf16 receive k_hat and v
    (ring=True: last min(L, S) tokens at slot pos mod S; ring=False: every token at slot pos)."""
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wk, "wk", torch.float32)
    B, L, Hkv, d = k.shape
    st = _lib.zg_kv_cache_write(_ptr(k), _ptr(v), _ptr(pos), _ptr(wk), _ptr(k_cache), _ptr(v_cache), B, L, Hkv, d,
                                int(k_cache.shape[2]), 1 if ring else 0, int(rotary_dim), float(theta), float(eps),
                                _stream(stream))
    _raise(st, "zg_kv_cache_write")


def kv_cache_write_fp8(k, v, pos, wk, k_cache, v_cache, *, ring, k_scale=1.0, v_scale=1.0, rotary_dim, theta,
                       eps=1e-6, stream=None):
    """kv_cache_write into E4M3 caches (float8_e4m3fn or uint8 [B,Hkv,S,d]): e4m3(k_hat * k_scale), e4m3(v * v_scale)."""
    for t, n in ((k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, 4)
    _check_cache(k_cache, "k_cache", True, 4)
    _check_cache(v_cache, "v_cache", True, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wk, "wk", torch.float32)
    B, L, Hkv, d = k.shape
    st = _lib.zg_kv_cache_write_fp8(_ptr(k), _ptr(v), _ptr(pos), _ptr(wk), _ptr(k_cache), _ptr(v_cache), B, L, Hkv,
                                    d, int(k_cache.shape[2]), 1 if ring else 0, int(rotary_dim), float(theta),
                                    float(eps), float(k_scale), float(v_scale), _stream(stream))
    _raise(st, "zg_kv_cache_write_fp8")


def linear(x, w, *, out=None, stream=None):
    """y = x @ w on the library's tensor-core GEMM: x [..., K], w [K, N] bf16 -> y [..., N] bf16."""
    _check(x, "x", torch.bfloat16)
    _check(w, "w", torch.bfloat16, 2)
    K, N = w.shape
    if x.shape[-1] != K:
        raise ValueError(f"x has {x.shape[-1]} columns, w has {K} rows")
    M = x.numel() // K
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    _check(out, "out", torch.bfloat16)
    _raise(_lib.zg_linear(_ptr(x), _ptr(w), _ptr(out), M, N, K, _stream(stream)), "zg_linear")
    return out


def gated_swa_layer_workspace_bytes(B, L, Hq, Hkv, d) -> int:
    return int(_lib.zg_gated_swa_layer_workspace_bytes(int(B), int(L), int(Hq), int(Hkv), int(d)))


def gated_swa_layer(h, w_q, w_k, w_v, w_g, w_o, pos, wq, wk, *, Hq, Hkv, window=128, rotary_dim, theta, eps=1e-6,
                    out=None, workspace=None, stream=None):
    """A whole gated SWA layer: y = o_proj(A_SWA(q, k, v) * sigmoid(g_proj(h))).
    h [B,L,hidden] bf16; w_q, w_g [hidden, Hq*d], w_k, w_v [hidden, Hkv*d], w_o [Hq*d, hidden] bf16
    (y = x W); pos [B,L] int32; wq, wk [d] float32.  Returns y [B,L,hidden] bf16."""
    _check(h, "h", torch.bfloat16, 3)
    for t, n in ((w_q, "w_q"), (w_k, "w_k"), (w_v, "w_v"), (w_g, "w_g"), (w_o, "w_o")):
        _check(t, n, torch.bfloat16, 2)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, hidden = h.shape
    d = w_q.shape[1] // Hq
    if out is None:
        out = torch.empty_like(h)
    _check(out, "out", torch.bfloat16, 3)
    need = gated_swa_layer_workspace_bytes(B, L, Hq, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=h.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_gated_swa_layer(_ptr(h), _ptr(w_q), _ptr(w_k), _ptr(w_v), _ptr(w_g), _ptr(w_o), _ptr(pos), _ptr(wq),
                                 _ptr(wk), _ptr(out), B, L, hidden, int(Hq), int(Hkv), d, int(window), int(rotary_dim),
                                 float(theta), float(eps), _ptr(workspace), ws_bytes, _stream(stream))
    _raise(st, "zg_gated_swa_layer")
    return out


def attention_backward_workspace_bytes(B, L, Hq, Hkv, d) -> int:
    return int(_lib.zg_attention_backward_workspace_bytes(int(B), int(L), int(Hq), int(Hkv), int(d)))


def attention_backward(q, k, v, gate, pos, wq, wk, dout, *, window, rotary_dim, theta, eps=1e-6, workspace=None,
                       stream=None):
    """Gradients of sum(out * dout) for the prefill out = swa_prefill(...) (gate given, window >= 1) or
    global_prefill(...) (gate None, window <= 0).  Inputs as the forward takes them, dout [B,L,Hq,d] bf16.
    Returns (dq, dk, dv, dgate) as float32 tensors, dgate None without a gate."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _check(t, n, torch.bfloat16, 4)
    if gate is not None:
        _check(gate, "gate", torch.bfloat16, 4)
    _check(pos, "pos", torch.int32, 2)
    _check(wq, "wq", torch.float32)
    _check(wk, "wk", torch.float32)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=q.device)
    dgate = torch.empty(q.shape, dtype=torch.float32, device=q.device) if gate is not None else None
    need = attention_backward_workspace_bytes(B, L, Hq, Hkv, d)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.zg_attention_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk), _ptr(dout),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dgate), B, L, Hq, Hkv, d, int(window),
                                    int(rotary_dim), float(theta), float(eps), _ptr(workspace), ws_bytes,
                                    _stream(stream))
    _raise(st, "zg_attention_backward")
    return dq, dk, dv, dgate


def hybrid_decode_workspace_bytes(NG, B, Hq, d, S_max) -> int:
    return int(_lib.zg_hybrid_decode_workspace_bytes(int(NG), int(B), int(Hq), int(d), int(S_max)))


def hybrid_decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, *,
                  rotary_dim, theta, eps=1e-6, out=None, workspace=None, stream=None):
    """One decode step through the hybrid layer stack (caches updated in place).
    q, gate [NL,B,Hq,d]; k_new, v_new [NL,B,Hkv,d]; pos [B] int32 (device); wq, wk [NL,d];
    is_global: sequence of NL flags (host); k_glob, v_glob [NG,B,Hkv,S,d]; k_ring, v_ring [NS,B,Hkv,W,d]."""
    return _decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, rotary_dim, theta,
                   eps, out, workspace, stream, fp8=False, k_scale=1.0, v_scale=1.0)


def hybrid_decode_fp8(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, *,
                      k_scale=1.0, v_scale=1.0, rotary_dim, theta, eps=1e-6, out=None, workspace=None, stream=None):
    """hybrid_decode over E4M3 caches (torch.float8_e4m3fn or uint8 tensors of the same shapes) holding
    e4m3(k_hat * k_scale) and e4m3(v * v_scale)."""
    return _decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, rotary_dim, theta,
                   eps, out, workspace, stream, fp8=True, k_scale=k_scale, v_scale=v_scale)


def _check_cache(t, name, fp8, ndim):
    if fp8:
        if t is None:
            raise ValueError(f"{name} is required")
        if t.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
            raise ValueError(f"{name} must be float8_e4m3fn or uint8, got {t.dtype}")
        _check(t, name, t.dtype, ndim)
    else:
        _check(t, name, torch.bfloat16, ndim)


def _decode(q, k_new, v_new, gate, pos, wq, wk, is_global, k_glob, v_glob, k_ring, v_ring, rotary_dim, theta, eps,
            out, workspace, stream, *, fp8, k_scale, v_scale):
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (gate, "gate")):
        _check(t, n, torch.bfloat16)
    _check(pos, "pos", torch.int32, 1)
    _check(wq, "wq", torch.float32, 2)
    _check(wk, "wk", torch.float32, 2)
    NL, B, Hq, d = q.shape
    Hkv = k_new.shape[2]
    flags = bytes(1 if int(x) else 0 for x in (is_global.tolist() if hasattr(is_global, "tolist") else is_global))
    NG = sum(flags)
    S = 0
    W = 0
    if NG:
        _check_cache(k_glob, "k_glob", fp8, 5)
        _check_cache(v_glob, "v_glob", fp8, 5)
        S = k_glob.shape[3]
    if NL - NG:
        _check_cache(k_ring, "k_ring", fp8, 5)
        _check_cache(v_ring, "v_ring", fp8, 5)
        W = k_ring.shape[3]
    else:
        W = 128
    if out is None:
        out = torch.empty_like(q)
    need = hybrid_decode_workspace_bytes(NG, B, Hq, d, S)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    flag_buf = ctypes.create_string_buffer(flags, len(flags))
    head = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(gate), _ptr(pos), _ptr(wq), _ptr(wk),
            ctypes.cast(flag_buf, ctypes.c_void_p), _ptr(k_glob), _ptr(v_glob), _ptr(k_ring), _ptr(v_ring), _ptr(out),
            NL, B, Hq, Hkv, d, int(S), int(W), int(rotary_dim), float(theta), float(eps))
    if fp8:
        st = _lib.zg_hybrid_decode_fp8(*head, float(k_scale), float(v_scale), _ptr(workspace), ws_bytes,
                                       _stream(stream))
        _raise(st, "zg_hybrid_decode_fp8")
    else:
        st = _lib.zg_hybrid_decode(*head, _ptr(workspace), ws_bytes, _stream(stream))
        _raise(st, "zg_hybrid_decode")
    return out


def device_status():
    """(status, detail): synchronises and reads/clears the device error word."""
    detail = ctypes.c_uint32(0)
    st = _lib.zg_device_status(ctypes.byref(detail))
    return st, detail.value


def selftest_bounded_wait(limit_ns: int, stream=None):
    _raise(_lib.zg_selftest_bounded_wait(int(limit_ns), _stream(stream)), "zg_selftest_bounded_wait")


def selftest_index_check(stream=None):
    _raise(_lib.zg_selftest_index_check(_stream(stream)), "zg_selftest_index_check")


def debug_build() -> bool:
    return bool(_lib.zg_debug_build())
