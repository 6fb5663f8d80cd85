"""The debug build: libzgattn_debug.so, the same kernels compiled with ZG_DEBUG, in which every
plain global-memory index (the TMA copies are bounds-checked by the hardware) is checked before
the access; an index out of range is recorded in the device error word and skipped.

The debug library runs in a child process (ZG_LIBRARY=debug selects it in the binding) on
small, odd shapes through every instrumented kernel -- gated SWA and global prefill, the k_hat
pre-pass, the E4M3 global and sliding-window prefills and their pre-passes, the tensor-core
backward (windowed and global), the decode step and its split merge (bf16 and E4M3 caches), the cache writer -- each
checked against the fp64 oracle with a clean error word.  Then the index check's own error
path is exercised without a fault (zg_selftest_index_check) and the context is shown to be
usable afterwards.  In the normal build the same self test records nothing."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, torch
import numpy as np
sys.path.insert(0, "tests")
import global_attention_fwd_b300 as zg
import oracle, workloads
from parity import assert_close, rows_of
assert zg.debug_build(), zg.LIB_PATH
torch.manual_seed(0)

def clean(what):
    st, detail = zg.device_status()
    assert st == 0, (what, st, hex(detail))

def rnd(*s, g):
    return torch.randn(*s, generator=g).bfloat16()

def prefill(B, L, Hq, Hkv, d, window, seed):
    g = torch.Generator().manual_seed(seed)
    x = dict(q=rnd(B, L, Hq, d, g=g), k=rnd(B, L, Hkv, d, g=g), v=rnd(B, L, Hkv, d, g=g),
             gate=rnd(B, L, Hq, d, g=g), pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
             wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))
    dx = {k: v.cuda() for k, v in x.items()}
    r = workloads.rotary_dim_for(d)
    rows = list(range(B * L))
    if window:
        out = zg.swa_prefill(dx["q"], dx["k"], dx["v"], dx["gate"], dx["pos"], dx["wq"], dx["wk"], window=window,
                             rotary_dim=r, theta=1e4)
    else:
        out = zg.global_prefill(dx["q"], dx["k"], dx["v"], dx["pos"], dx["wq"], dx["wk"], rotary_dim=r, theta=1e4)
    torch.cuda.synchronize()
    clean(f"prefill {B} {L} {Hq}/{Hkv} d{d} W{window}")
    ref = oracle.prefill_rows(x["q"], x["k"], x["v"], x["gate"] if window else None, x["pos"], x["wq"], x["wk"],
                              window=window, rotary_dim=r, theta=1e4, eps=1e-6, rows=rows)
    assert_close(rows_of(out, rows), ref, f"debug prefill {B} {L} {Hq}/{Hkv} d{d} W{window}")
    if window:  # the cache writer over the same keys: a 40-slot ring
        kr = torch.zeros(B, Hkv, 40, d, dtype=torch.bfloat16, device="cuda")
        vr = torch.zeros_like(kr)
        zg.kv_cache_write(dx["k"], dx["v"], dx["pos"], dx["wk"], kr, vr, ring=True, rotary_dim=r, theta=1e4)
        torch.cuda.synchronize()
        clean("cache writer")
        i = L - 1
        assert torch.equal(vr[0, 0, i % 40].cpu(), x["v"][0, i, 0])

prefill(2, 33, 4, 1, 64, 37, 1)        # GQA 4, ragged tail, odd window
prefill(1, 170, 32, 2, 128, 128, 2)    # GQA 16
prefill(1, 91, 2, 2, 128, 5, 3)        # MHA
prefill(2, 77, 8, 2, 64, 0, 4)         # global, d = 64
prefill(1, 130, 32, 8, 128, 0, 5)      # global, GQA 4

def prefill_e4m3(B, L, Hq, Hkv, seed):  # global prefill on E4M3 inputs (k_hat and V^T pre-passes)
    g = torch.Generator().manual_seed(seed)
    st = {n: workloads.to_e4m3(rnd(B, L, h, 128, g=g), 1.0).view(torch.uint8) for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv))}
    deq = {n: st[n].view(torch.float8_e4m3fn).double() for n in st}
    pos = torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous()
    wq, wk = 0.5 + torch.rand(128, generator=g), 0.5 + torch.rand(128, generator=g)
    out = zg.global_prefill_fp8(st["q"].cuda(), st["k"].cuda(), st["v"].cuda(), pos.cuda(), wq.cuda(), wk.cuda(),
                                rotary_dim=42, theta=1e6)
    torch.cuda.synchronize()
    clean(f"e4m3 global prefill {B} {L} {Hq}/{Hkv}")
    rows = list(range(B * L))
    ref = oracle.prefill_rows(deq["q"], deq["k"], deq["v"], None, pos, wq, wk, window=0, rotary_dim=42, theta=1e6,
                              eps=1e-6, rows=rows)
    got = rows_of(out, rows)
    err = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert err <= 0.10, err  # the E4M3 path's own bound

prefill_e4m3(2, 45, 8, 2, 9)      # ragged: 45 keys, V^T padded to 48
prefill_e4m3(1, 200, 16, 1, 10)   # GQA 16

def swa_e4m3(B, L, Hq, Hkv, W, seed):  # gated sliding window on E4M3 inputs (the global pipeline's window mode)
    g = torch.Generator().manual_seed(seed)
    st = {n: workloads.to_e4m3(rnd(B, L, h, 128, g=g), 1.0).view(torch.uint8) for n, h in (("q", Hq), ("k", Hkv), ("v", Hkv))}
    deq = {n: st[n].view(torch.float8_e4m3fn).double() for n in st}
    gate = rnd(B, L, Hq, 128, g=g)
    pos = torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous()
    wq, wk = 0.5 + torch.rand(128, generator=g), 0.5 + torch.rand(128, generator=g)
    out = zg.swa_prefill_fp8(st["q"].cuda(), st["k"].cuda(), st["v"].cuda(), gate.cuda(), pos.cuda(), wq.cuda(), wk.cuda(),
                             window=W, rotary_dim=42, theta=1e4)
    torch.cuda.synchronize()
    clean(f"e4m3 swa prefill {B} {L} {Hq}/{Hkv} W{W}")
    rows = list(range(B * L))
    ref = oracle.prefill_rows(deq["q"], deq["k"], deq["v"], gate.double(), pos, wq, wk, window=W, rotary_dim=42,
                              theta=1e4, eps=1e-6, rows=rows)
    got = rows_of(out, rows)
    err = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert err <= 0.10, err

swa_e4m3(2, 150, 8, 2, 37, 11)    # odd window, two sequences
swa_e4m3(2, 2500, 16, 4, 128, 12)  # 320 work items: two or three per persistent CTA

from oracle import backward as bw

def backward(B, L, Hq, Hkv, W, gated, seed):  # the tensor-core backward (windowed, or the global layer for W = 0)
    g = torch.Generator().manual_seed(seed)
    x = dict(q=rnd(B, L, Hq, 128, g=g), k=rnd(B, L, Hkv, 128, g=g), v=rnd(B, L, Hkv, 128, g=g),
             gate=rnd(B, L, Hq, 128, g=g) if gated else None, dout=rnd(B, L, Hq, 128, g=g),
             pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
             wq=0.5 + torch.rand(128, generator=g), wk=0.5 + torch.rand(128, generator=g))
    d = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    got = zg.attention_backward(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], d["dout"], window=W,
                                rotary_dim=42, theta=1e4)
    torch.cuda.synchronize()
    clean(f"backward {B} {L} {Hq}/{Hkv} W{W}")
    ref = bw.gradients(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], x["dout"], window=W, rotary_dim=42,
                       theta=1e4, eps=1e-6)
    for n, a, r in zip(("dq", "dk", "dv", "dgate"), got, ref):
        if r is None:
            continue
        a = a.double().cpu().numpy(); r = r.detach().double().numpy()
        rel = float(np.linalg.norm(a - r) / np.linalg.norm(r))
        assert rel <= 1e-2, (n, rel)  # the tensor-core path's bar

backward(1, 170, 8, 2, 128, True, 12)   # windowed, ragged last tile
backward(1, 300, 4, 1, 0, False, 13)    # the global layer: three key blocks

def decode(flags, B, Hq, Hkv, d, S, W, positions, seed, fp8):
    g = torch.Generator().manual_seed(seed)
    NL, NG = len(flags), sum(flags)
    x = dict(q=rnd(NL, B, Hq, d, g=g), k_new=rnd(NL, B, Hkv, d, g=g), v_new=rnd(NL, B, Hkv, d, g=g),
             gate=rnd(NL, B, Hq, d, g=g), wq=0.5 + torch.rand(NL, d, generator=g), wk=0.5 + torch.rand(NL, d, generator=g),
             k_glob=rnd(NG, B, Hkv, S, d, g=g), v_glob=rnd(NG, B, Hkv, S, d, g=g),
             k_ring=rnd(NL - NG, B, Hkv, W, d, g=g), v_ring=rnd(NL - NG, B, Hkv, W, d, g=g))
    if fp8:
        for k in ("k_glob", "v_glob", "k_ring", "v_ring"):
            x[k] = workloads.to_e4m3(x[k], 1.0)
    host = {k: v.clone() for k, v in x.items()}
    dx = {k: v.cuda() for k, v in x.items()}
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    r = workloads.rotary_dim_for(d)
    f = zg.hybrid_decode_fp8 if fp8 else zg.hybrid_decode
    out = f(dx["q"], dx["k_new"], dx["v_new"], dx["gate"], pos, dx["wq"], dx["wk"], flags, dx["k_glob"], dx["v_glob"],
            dx["k_ring"], dx["v_ring"], rotary_dim=r, theta=1e6)
    torch.cuda.synchronize()
    clean(f"decode fp8={fp8}")
    for b, p in enumerate(positions):
        c = {k: (host[k][:, b].to(torch.bfloat16) if fp8 else host[k][:, b]) for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
        ref, _ = oracle.decode_seq(host["q"][:, b], host["k_new"][:, b], host["v_new"][:, b], host["gate"][:, b],
                                   host["wq"], host["wk"], flags, c["k_glob"], c["v_glob"], c["k_ring"], c["v_ring"],
                                   p=p, rotary_dim=r, theta=1e6, eps=1e-6)
        assert_close(out[:, b].double().cpu().numpy(), ref, f"debug decode fp8={fp8} seq {b}")

decode([0, 1, 0], 3, 12, 4, 128, 8300, 40, [8299, 3, 100], 6, False)   # GQA 3, two splits, 40-slot rings
decode([1, 0], 2, 16, 1, 64, 300, 128, [299, 0], 7, True)              # GQA 16, d = 64, E4M3 caches

# the index check's own error path, without an out-of-range access
zg.selftest_index_check()
st, detail = zg.device_status()
assert st == -10 and (detail >> 8) == 98 and (detail & 0xFF) == 5, (st, hex(detail))
assert zg.device_status()[0] == 0
prefill(1, 40, 4, 1, 64, 128, 8)  # the context is still usable
print("DEBUG_BUILD_OK")
'''


def _debug_lib():
    path = os.path.join(ROOT, "global_attention_fwd_b300", "libzgattn_debug.so")
    if not os.path.exists(path):
        subprocess.check_call([sys.executable, os.path.join(ROOT, "global_attention_fwd_b300", "_build.py"), "--debug"])
    return path


def test_debug_build_small_odd_shapes_and_index_check():
    _debug_lib()
    env = dict(os.environ, ZG_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "DEBUG_BUILD_OK" in r.stdout, (r.stdout[-3000:], r.stderr[-3000:])


def test_normal_build_index_selftest_records_nothing():
    import global_attention_fwd_b300 as zg

    assert not zg.debug_build()
    zg.device_status()
    zg.selftest_index_check()
    assert zg.device_status() == (0, 0)
