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
    assert _swa(zg, Hq=12, Hkv=1) == -4
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
    assert _glob(zg, d=64, rot=20) == -4
    assert _glob(zg, Hq=16) == -4
    assert _glob(zg, L=0) == 0
    assert _glob(zg, ws=None) == -6
    assert _glob(zg, ws_bytes=16 * 8 * 128 * 2 - 1) == -6
    assert _glob(zg, ws=A + 8) == -6
    assert zg.global_prefill_workspace_bytes(1, 16, 8, 128) == 16 * 8 * 128 * 2


def test_status_strings(zg):
    for s in range(-9, 1):
        assert zg.lib.zg_status_string(s)
    assert zg.lib.zg_status_string(-8) == b"device-side wait timed out"
