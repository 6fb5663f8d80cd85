"""zg_hybrid_decode_noalloc: the decode step for callers that cannot allocate
device memory (for instance a plugin whose host application owns all device
allocations, or a serving loop that must not allocate mid-request).  The
scratch comes from a fixed array inside the library.  Checked through the C ABI
against zg_hybrid_decode (caller workspace) on two calls in a row with
different sizes, so stale scratch contents from the first call would show in
the second.  Both run the same kernels on the same inputs, so the outputs must
be bit-identical; the first call is also checked against the fp64 oracle.  A
bad call must get the same status from both entry points.  This file is
collected last on purpose."""
import ctypes

import pytest
import torch

import oracle
from parity import assert_close

pytestmark = pytest.mark.gpu

P, I, I64, D, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_float, ctypes.c_size_t


@pytest.fixture(scope="module")
def lib():
    import global_attention_fwd_b300 as zg
    lib = zg.lib
    lib.zg_hybrid_decode_noalloc.argtypes = [P] * 13 + [I] * 5 + [I64, I, I, D, F, P]
    lib.zg_hybrid_decode_noalloc.restype = I
    return lib


def _case(NL, flags, B, Hq, Hkv, S, seed):
    g = torch.Generator().manual_seed(seed)
    d, W = 128, 128
    NG = sum(flags)

    def r(*s):
        return torch.randn(*s, generator=g).bfloat16().cuda()

    return dict(q=r(NL, B, Hq, d), k_new=r(NL, B, Hkv, d), v_new=r(NL, B, Hkv, d), gate=r(NL, B, Hq, d),
                wq=(0.5 + torch.rand(NL, d, generator=g)).cuda(), wk=(0.5 + torch.rand(NL, d, generator=g)).cuda(),
                k_glob=r(NG, B, Hkv, S, d), v_glob=r(NG, B, Hkv, S, d), k_ring=r(NL - NG, B, Hkv, W, d),
                v_ring=r(NL - NG, B, Hkv, W, d))


def _call(lib, x, flags, pos, S, noalloc):
    NL, B, Hq, d = x["q"].shape
    Hkv = x["k_new"].shape[2]
    out = torch.empty_like(x["q"])
    fl = ctypes.create_string_buffer(bytes(flags), len(flags))
    pos_t = torch.tensor(pos, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    args = [ptr(x["q"]), ptr(x["k_new"]), ptr(x["v_new"]), ptr(x["gate"]), ptr(pos_t), ptr(x["wq"]), ptr(x["wk"]),
            ctypes.cast(fl, ctypes.c_void_p), ptr(x["k_glob"]), ptr(x["v_glob"]), ptr(x["k_ring"]), ptr(x["v_ring"]),
            ptr(out), NL, B, Hq, Hkv, d, S, 128, 42, 1e6, 1e-6]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        st = lib.zg_hybrid_decode_noalloc(*args, stream)
    else:
        need = lib.zg_hybrid_decode_workspace_bytes(sum(flags), B, Hq, d, S)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        st = lib.zg_hybrid_decode(*args, ptr(ws), need, stream)
    torch.cuda.synchronize()
    assert st == 0, st
    return out


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    # call 1: 3 global layers, 9000-slot caches (3 splits); call 2: 1 global layer, 5000 slots (2 splits)
    for i, (flags, B, S, pos, seed) in enumerate((([0, 1, 0, 1, 1, 0], 3, 9000, [8999, 4096, 60], 1),
                                                  ([1, 0, 0], 2, 5000, [4000, 127], 2))):
        x = _case(len(flags), flags, B, 32, 8, S, seed)
        before = {k: x[k].clone() for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
        ref = _call(lib, x, flags, pos, S, noalloc=False)
        # the step wrote the new token's cache slots; give the second call the caches as they were
        after = {k: x[k].clone() for k in before}
        for k in before:
            x[k].copy_(before[k])
        got = _call(lib, x, flags, pos, S, noalloc=True)
        assert torch.equal(got, ref), f"call {i}: allocation-free output differs from the workspace decode"
        for k in before:
            assert torch.equal(x[k], after[k]), f"call {i}: cache {k} differs"
        if i == 0:
            b = 0
            want, _ = oracle.decode_seq(x["q"][:, b].cpu(), x["k_new"][:, b].cpu(), x["v_new"][:, b].cpu(),
                                        x["gate"][:, b].cpu(), x["wq"].cpu(), x["wk"].cpu(), flags,
                                        before["k_glob"][:, b].cpu(), before["v_glob"][:, b].cpu(),
                                        before["k_ring"][:, b].cpu(), before["v_ring"][:, b].cpu(), p=pos[b],
                                        rotary_dim=42, theta=1e6, eps=1e-6)
            assert_close(got[:, b].double().cpu().numpy(), want, "allocation-free decode vs oracle")


def _raw(lib, x, flags, pos_t, out, NL, B, Hq, Hkv, d, S, window, noalloc, ws=None, ws_bytes=0):
    fl = ctypes.create_string_buffer(bytes(flags), max(1, len(flags)))
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    args = [ptr(x["q"]), ptr(x["k_new"]), ptr(x["v_new"]), ptr(x["gate"]), ptr(pos_t), ptr(x["wq"]), ptr(x["wk"]),
            ctypes.cast(fl, ctypes.c_void_p), ptr(x["k_glob"]), ptr(x["v_glob"]), ptr(x["k_ring"]), ptr(x["v_ring"]),
            ptr(out), NL, B, Hq, Hkv, d, S, window, 42, 1e6, 1e-6]
    if noalloc:
        return lib.zg_hybrid_decode_noalloc(*args, None)
    return lib.zg_hybrid_decode(*args, ptr(ws), ws_bytes, None)


def test_noalloc_reports_argument_errors_like_the_workspace_entry_point(lib):
    flags = [1, 0]
    x = _case(2, flags, 2, 32, 8, 256, 4)
    pos = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.empty_like(x["q"])
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    bad = [
        dict(d=96),                   # a head size the kernels do not implement
        dict(Hq=30),                  # Hq not a multiple of Hkv
        dict(NL=200),                 # more layers than a call takes
        dict(window=0),               # empty window
        dict(S=0),                    # global layers without cache slots
    ]
    for change in bad:
        a = dict(NL=2, B=2, Hq=32, Hkv=8, d=128, S=256, window=128)
        a.update(change)
        fl = flags if a["NL"] == 2 else [0] * a["NL"]
        st_ws = _raw(lib, x, fl, pos, out, a["NL"], a["B"], a["Hq"], a["Hkv"], a["d"], a["S"], a["window"],
                     noalloc=False, ws=ws, ws_bytes=ws.numel())
        st_na = _raw(lib, x, fl, pos, out, a["NL"], a["B"], a["Hq"], a["Hkv"], a["d"], a["S"], a["window"],
                     noalloc=True)
        assert st_ws < 0 and st_ws == st_na, (change, st_ws, st_na)
    # a NULL pointer
    y = dict(x, q=None)
    assert _raw(lib, y, flags, pos, out, 2, 2, 32, 8, 128, 256, 128, noalloc=True) == -1


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    flags = [1] * 5
    x = _case(5, flags, 1, 32, 8, 16, 3)
    # 5 layers x 64 sequences x 32 heads with 262144 slots would need ~341 MB of scratch
    NL, B, Hq, Hkv, d, S = 5, 64, 32, 8, 128, 262144
    need = lib.zg_hybrid_decode_workspace_bytes(NL, B, Hq, d, S)
    assert need > (64 << 20)
    fl = ctypes.create_string_buffer(bytes(flags), 5)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    pos = torch.zeros(B, dtype=torch.int32, device="cuda")
    st = lib.zg_hybrid_decode_noalloc(ptr(x["q"]), ptr(x["k_new"]), ptr(x["v_new"]), ptr(x["gate"]), ptr(pos),
                                      ptr(x["wq"]), ptr(x["wk"]), ctypes.cast(fl, ctypes.c_void_p), ptr(x["k_glob"]),
                                      ptr(x["v_glob"]), ptr(x["k_ring"]), ptr(x["v_ring"]), ptr(x["q"]), NL, B, Hq,
                                      Hkv, d, S, 128, 42, 1e6, 1e-6, None)
    assert st == -6
