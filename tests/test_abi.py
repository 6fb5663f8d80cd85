"""The C ABI without a GPU: the library loads, exports every entry point that
include/zg_attn.h declares, and rejects bad arguments on the host before it
launches anything (these calls return before any CUDA call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zg_attn.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zg_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("zg_swa_prefill", "zg_global_prefill", "zg_hybrid_decode", "zg_hybrid_decode_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(zg):
    lib = ctypes.CDLL(zg.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared()) == set(zg.EXPORTS)


def test_debug_library_exports_the_same_symbols(zg):
    path = os.path.join(os.path.dirname(zg.LIB_PATH), "libzgattn_debug.so")
    if not os.path.exists(path):
        pytest.skip("debug library not built")
    dbg = ctypes.CDLL(path)
    missing = [n for n in _declared() if not hasattr(dbg, n)]
    assert not missing, missing
    assert dbg.zg_debug_build() == 1
    assert zg.lib.zg_debug_build() == 0


A = 1 << 20  # a fake, 16-byte aligned, non-null address (never dereferenced: validation fails first)


def _swa(zg, **kw):
    a = dict(q=A, k=A, v=A, gate=A, pos=A, wq=A, wk=A, out=A, B=1, L=16, Hq=4, Hkv=1, d=64, window=128,
             rot=20, theta=1e4, eps=1e-6)
    a.update(kw)
    return zg.lib.zg_swa_prefill(a["q"], a["k"], a["v"], a["gate"], a["pos"], a["wq"], a["wk"], a["out"], a["B"],
                                 a["L"], a["Hq"], a["Hkv"], a["d"], a["window"], a["rot"], a["theta"], a["eps"], None)


def test_swa_rejects_bad_arguments_before_launch(zg):
    assert _swa(zg, q=None) == -1
    assert _swa(zg, gate=None) == -1
    assert _swa(zg, k=A + 8) == -2
    assert _swa(zg, out=A + 2) == -2
    assert _swa(zg, B=-1) == -3
    assert _swa(zg, Hq=6, Hkv=4) == -3
    assert _swa(zg, rot=21) == -3
    assert _swa(zg, rot=66) == -3
    assert _swa(zg, window=0) == -3
    assert _swa(zg, theta=0.0) == -3
    assert _swa(zg, eps=-1.0) == -3
    assert _swa(zg, window=129) == -4
    assert _swa(zg, d=96, rot=30) == -4
    assert _swa(zg, Hq=12, Hkv=1) == -4   # G must divide 128
    assert _swa(zg, Hq=32, Hkv=1) == -4   # G > 16
    # empty inputs are a no-op
    assert _swa(zg, L=0) == 0
    assert _swa(zg, B=0) == 0


def _glob(zg, **kw):
    a = dict(q=A, k=A, v=A, pos=A, wq=A, wk=A, out=A, B=1, L=16, Hq=32, Hkv=8, d=128, rot=42, theta=1e6, eps=1e-6)
    a.update(kw)
    return zg.lib.zg_global_prefill(a["q"], a["k"], a["v"], a["pos"], a["wq"], a["wk"], a["out"], a["B"], a["L"],
                                    a["Hq"], a["Hkv"], a["d"], a["rot"], a["theta"], a["eps"], a.get("ws", A),
                                    a.get("ws_bytes", 1 << 40), None)


def test_global_rejects_bad_arguments_before_launch(zg):
    assert _glob(zg, v=None) == -1
    assert _glob(zg, pos=A + 4) == -2
    assert _glob(zg, L=-5) == -3
    assert _glob(zg, d=96, rot=30) == -4
    assert _glob(zg, Hq=24) == -4          # G = 3 does not divide 128
    assert _glob(zg, L=0) == 0
    assert _glob(zg, ws=None) == -6
    assert _glob(zg, ws_bytes=16 * 8 * 128 * 2 - 1) == -6
    assert _glob(zg, ws=A + 8) == -6
    assert zg.global_prefill_workspace_bytes(1, 16, 8, 128) == 16 * 8 * 128 * 2


def test_status_strings(zg):
    for s in range(-10, 1):
        assert zg.lib.zg_status_string(s)
    assert zg.lib.zg_status_string(-8) == b"device-side wait timed out"


def _swa_cache(zg, **kw):
    a = dict(q=A, k=A, v=A, gate=A, pos=A, wq=A, wk=A, out=A, B=1, L=16, Hq=32, Hkv=8, d=128, window=128,
             rot=42, theta=1e6, eps=1e-6, kr=A, vr=A, slots=128)
    a.update(kw)
    return zg.lib.zg_swa_prefill_with_cache(a["q"], a["k"], a["v"], a["gate"], a["pos"], a["wq"], a["wk"], a["out"],
                                            a["B"], a["L"], a["Hq"], a["Hkv"], a["d"], a["window"], a["rot"],
                                            a["theta"], a["eps"], a["kr"], a["vr"], a["slots"], None)


def _glob_cache(zg, **kw):
    a = dict(q=A, k=A, v=A, pos=A, wq=A, wk=A, out=A, B=1, L=16, Hq=32, Hkv=8, d=128, rot=42, theta=1e6, eps=1e-6,
             ws=A, ws_bytes=1 << 30, kc=A, vc=A, smax=4096)
    a.update(kw)
    return zg.lib.zg_global_prefill_with_cache(a["q"], a["k"], a["v"], a["pos"], a["wq"], a["wk"], a["out"], a["B"],
                                               a["L"], a["Hq"], a["Hkv"], a["d"], a["rot"], a["theta"], a["eps"],
                                               a["ws"], a["ws_bytes"], a["kc"], a["vc"], a["smax"], None)


def test_prefill_with_cache_rejects_bad_cache_arguments_before_launch(zg):
    # cache arguments are checked first; nothing (not even the prefill) is launched on failure
    assert _swa_cache(zg, kr=None) == -1
    assert _swa_cache(zg, vr=A + 4) == -2
    assert _swa_cache(zg, slots=0) == -3
    assert _swa_cache(zg, d=96, rot=30) == -4      # decode caches have d = 64 or 128
    assert _swa_cache(zg, q=None) == -1            # then the prefill's own checks
    assert _swa_cache(zg, window=0) == -3
    assert _glob_cache(zg, vc=None) == -1
    assert _glob_cache(zg, kc=A + 8) == -2
    assert _glob_cache(zg, smax=0) == -3
    assert _glob_cache(zg, ws=None) == -6
    assert _glob_cache(zg, Hq=24) == -4
    assert _glob_cache(zg, d=96, rot=30) == -4


def test_kv_cache_write_rejects_bad_arguments(zg):
    def call(**kw):
        a = dict(k=A, v=A, pos=A, wk=A, kc=A, vc=A, B=1, L=16, Hkv=8, d=128, S=128, ring=1, rot=42, theta=1e6,
                 eps=1e-6)
        a.update(kw)
        return zg.lib.zg_kv_cache_write(a["k"], a["v"], a["pos"], a["wk"], a["kc"], a["vc"], a["B"], a["L"], a["Hkv"],
                                        a["d"], a["S"], a["ring"], a["rot"], a["theta"], a["eps"], None)
    assert call(k=None) == -1
    assert call(kc=None) == -1
    assert call(pos=A + 4) == -2
    assert call(S=0) == -3
    assert call(ring=2) == -3
    assert call(rot=43) == -3
    assert call(d=96, rot=30) == -4


def test_gated_swa_layer_rejects_bad_arguments(zg):
    def call(**kw):
        a = dict(h=A, wq_=A, wk_=A, wv_=A, wg_=A, wo_=A, pos=A, wq=A, wk=A, y=A, B=1, L=16, hidden=4096, Hq=32, Hkv=8,
                 d=128, window=128, rot=42, theta=1e6, eps=1e-6, ws=A, ws_bytes=1 << 40)
        a.update(kw)
        return zg.lib.zg_gated_swa_layer(a["h"], a["wq_"], a["wk_"], a["wv_"], a["wg_"], a["wo_"], a["pos"], a["wq"],
                                         a["wk"], a["y"], a["B"], a["L"], a["hidden"], a["Hq"], a["Hkv"], a["d"],
                                         a["window"], a["rot"], a["theta"], a["eps"], a["ws"], a["ws_bytes"], None)
    assert call(wo_=None) == -1
    assert call(pos=None) == -1
    assert call(wg_=A + 2) == -2
    assert call(hidden=4100) == -3
    assert call(Hq=30) == -3
    assert call(window=0) == -3
    assert call(d=96, rot=20) == -4
    assert call(ws=None) == -6
    assert call(ws_bytes=1024) == -6
    assert call(rot=130) == -3                # rotary_dim > d
    assert call(rot=80) == -4                 # the fused epilogue takes rotary_dim <= 64
    # q_hat, k_hat, v, sigmoid(g), a: (Hq + Hkv + Hkv + Hq + Hq) * d * 2 bytes per token, 256-byte aligned
    assert zg.gated_swa_layer_workspace_bytes(1, 16, 32, 8, 128) == 16 * (32 * 3 + 8 * 2) * 128 * 2


def test_linear_rejects_bad_arguments(zg):
    def call(**kw):
        a = dict(x=A, w=A, y=A, M=64, N=256, K=128)
        a.update(kw)
        return zg.lib.zg_linear(a["x"], a["w"], a["y"], a["M"], a["N"], a["K"], None)
    assert call(w=None) == -1
    assert call(y=A + 8) == -2
    assert call(N=100) == -3    # rows of W must be 16-byte multiples
    assert call(K=0) == -3
    assert call(M=-1) == -3
    assert call(M=0) == 0       # nothing to do, nothing launched


def test_attention_backward_rejects_bad_arguments(zg):
    def call(**kw):
        a = dict(q=A, k=A, v=A, gate=A, pos=A, wq=A, wk=A, dout=A, dq=A, dk=A, dv=A, dg=A, B=1, L=16, Hq=32, Hkv=8,
                 d=128, window=128, rot=42, theta=1e4, eps=1e-6, ws=A, ws_bytes=1 << 40)
        a.update(kw)
        return zg.lib.zg_attention_backward(a["q"], a["k"], a["v"], a["gate"], a["pos"], a["wq"], a["wk"], a["dout"],
                                            a["dq"], a["dk"], a["dv"], a["dg"], a["B"], a["L"], a["Hq"], a["Hkv"],
                                            a["d"], a["window"], a["rot"], a["theta"], a["eps"], a["ws"],
                                            a["ws_bytes"], None)
    assert call(dout=None) == -1
    assert call(dv=None) == -1
    assert call(dg=None) == -1            # a gate needs its gradient
    assert call(gate=None) == -3          # and no gate, no gate gradient
    assert call(dq=A + 4) == -2
    assert call(gate=A + 8) == -2
    assert call(Hq=30) == -3
    assert call(rot=41) == -3
    assert call(eps=-1.0) == -3
    assert call(d=64, rot=20) == -4
    assert call(ws=None) == -6
    assert call(ws_bytes=1024) == -6
    assert call(B=0) == 0 and call(L=0) == 0  # nothing to do, nothing launched
    # fp32 q_hat, dA, dq_hat per query row, k_hat, dk_hat per key row, three floats per query row
    assert zg.attention_backward_workspace_bytes(2, 16, 32, 8, 128) == 4 * (2 * 16 * (32 * 128 * 3 + 32 * 3 + 8 * 128 * 2))
    assert zg.attention_backward_workspace_bytes(2, 16, 32, 8, 64) == 0


def test_fp8_entry_points_reject_bad_arguments(zg):
    def dec(**kw):
        a = dict(q=A, kn=A, vn=A, g=A, pos=A, wq=A, wk=A, flags=None, kg=A, vg=A, kr=A, vr=A, out=A, NL=2, B=1, Hq=4,
                 Hkv=1, d=128, S=256, W=128, rot=42, theta=1e6, eps=1e-6, ks=1.0, vs=8.0, ws=A, wsb=1 << 40)
        a.update(kw)
        flags = ctypes.create_string_buffer(b"\x00\x01", 2)
        return zg.lib.zg_hybrid_decode_fp8(a["q"], a["kn"], a["vn"], a["g"], a["pos"], a["wq"], a["wk"],
                                           ctypes.cast(flags, ctypes.c_void_p), a["kg"], a["vg"], a["kr"], a["vr"],
                                           a["out"], a["NL"], a["B"], a["Hq"], a["Hkv"], a["d"], a["S"], a["W"],
                                           a["rot"], a["theta"], a["eps"], a["ks"], a["vs"], a["ws"], a["wsb"], None)
    assert dec(ks=0.0) == -3
    assert dec(vs=float("inf")) == -3
    assert dec(kg=None) == -1
    assert dec(vr=A + 8) == -2
    assert dec(d=96, rot=30) == -4
    assert dec(Hq=17, Hkv=1) == -4   # more than 16 query heads per KV head
    assert dec(W=0) == -3

    def wr(**kw):
        a = dict(k=A, v=A, pos=A, wk=A, kc=A, vc=A, B=1, L=16, Hkv=8, d=128, S=128, ring=1, rot=42, theta=1e6,
                 eps=1e-6, ks=1.0, vs=8.0)
        a.update(kw)
        return zg.lib.zg_kv_cache_write_fp8(a["k"], a["v"], a["pos"], a["wk"], a["kc"], a["vc"], a["B"], a["L"],
                                            a["Hkv"], a["d"], a["S"], a["ring"], a["rot"], a["theta"], a["eps"],
                                            a["ks"], a["vs"], None)
    assert wr(kc=None) == -1
    assert wr(ks=-1.0) == -3
    assert wr(vs=float("nan")) == -3
    assert wr(S=0) == -3
