"""Prefill that also writes the decode caches: cache contents against the oracle's
normalised, rotated keys, and prefill -> decode end to end against the oracle's
prefill of the longer sequence."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close

pytestmark = pytest.mark.gpu

D, HQ, HKV, R, THETA, EPS = 128, 32, 8, 42, 1e6, 1e-6
SENTINEL = 7.0  # cache slots a prefill must not touch keep this value


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _inputs(B, L, seed, pos0=(0,), d=D, Hq=HQ, Hkv=HKV):
    g = torch.Generator().manual_seed(seed)
    pos = torch.stack([torch.arange(L, dtype=torch.int32) + int(pos0[b % len(pos0)]) for b in range(B)]).contiguous()
    return dict(q=torch.randn(B, L, Hq, d, generator=g).bfloat16(), k=torch.randn(B, L, Hkv, d, generator=g).bfloat16(),
                v=torch.randn(B, L, Hkv, d, generator=g).bfloat16(), gate=torch.randn(B, L, Hq, d, generator=g).bfloat16(),
                pos=pos, wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))


def _khat(inp, b, i, g):
    """oracle k_hat of token i, KV head g of sequence b (fp64)"""
    x = inp["k"][b, i, g].double().numpy()
    xn = oracle.rmsnorm(x, inp["wk"].double().numpy(), EPS)
    return oracle.rope(xn, R, int(inp["pos"][b, i]), THETA)


def _check_slot(ck, cv, inp, b, g, slot, i, what):
    got = ck[b, g, slot].double().cpu().numpy()
    ref = _khat(inp, b, i, g)
    # bf16 rounding of the stored key: half an ulp of 2^-8 relative, plus fp32 arithmetic
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5), (what, b, g, slot, np.abs(got - ref).max())
    assert torch.equal(cv[b, g, slot].cpu(), inp["v"][b, i, g]), (what, b, g, slot)


@pytest.mark.parametrize("L,pos0", [(300, (0, 1000)), (50, (0, 77))])
def test_swa_prefill_writes_the_ring(zg, L, pos0):
    B, W = 2, 128
    inp = _inputs(B, L, seed=L, pos0=pos0)
    d = {k: v.cuda() for k, v in inp.items()}
    kr = torch.full((B, HKV, W, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    vr = kr.clone()
    out = zg.swa_prefill_with_cache(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], kr, vr,
                                    window=W, rotary_dim=R, theta=THETA, eps=EPS)
    plain = zg.swa_prefill(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], window=W, rotary_dim=R,
                           theta=THETA, eps=EPS)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    assert torch.equal(out, plain)  # the prefill itself is unchanged
    written = set()
    for b in range(B):
        for i in range(max(0, L - W), L):
            slot = int(inp["pos"][b, i]) % W
            written.add((b, slot))
            for g in (0, 3, 7):
                _check_slot(kr, vr, inp, b, g, slot, i, "ring")
    for b in range(B):
        for slot in range(W):
            if (b, slot) not in written:
                assert bool((kr[b, :, slot] == SENTINEL).all()) and bool((vr[b, :, slot] == SENTINEL).all())


def test_global_prefill_writes_the_cache(zg):
    B, L, S = 2, 200, 256
    inp = _inputs(B, L, seed=3)
    d = {k: v.cuda() for k, v in inp.items()}
    kc = torch.full((B, HKV, S, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    out = zg.global_prefill_with_cache(d["q"], d["k"], d["v"], d["pos"], d["wq"], d["wk"], kc, vc, rotary_dim=R,
                                       theta=THETA, eps=EPS)
    plain = zg.global_prefill(d["q"], d["k"], d["v"], d["pos"], d["wq"], d["wk"], rotary_dim=R, theta=THETA, eps=EPS)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    assert torch.equal(out, plain)
    for b in range(B):
        for i in list(range(0, L, 13)) + [L - 1]:
            for g in (0, 5):
                _check_slot(kc, vc, inp, b, g, int(inp["pos"][b, i]), i, "global")
    assert bool((kc[:, :, L:] == SENTINEL).all()) and bool((vc[:, :, L:] == SENTINEL).all())


def test_standalone_writer_matches_the_prefill_call(zg):
    B, L, W = 2, 200, 128
    inp = _inputs(B, L, seed=6, pos0=(5, 300))
    d = {k: v.cuda() for k, v in inp.items()}
    kr = torch.full((B, HKV, W, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    vr = kr.clone()
    kr2, vr2 = kr.clone(), vr.clone()
    zg.swa_prefill_with_cache(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], kr, vr, window=W,
                              rotary_dim=R, theta=THETA, eps=EPS)
    zg.kv_cache_write(d["k"], d["v"], d["pos"], d["wk"], kr2, vr2, ring=True, rotary_dim=R, theta=THETA, eps=EPS)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    assert torch.equal(kr, kr2) and torch.equal(vr, vr2)


def test_position_without_a_slot_is_reported(zg):
    B, L, S = 1, 40, 32  # positions 32..39 have no slot in a 32-slot global cache
    inp = _inputs(B, L, seed=4)
    d = {k: v.cuda() for k, v in inp.items()}
    kc = torch.full((B, HKV, S, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    zg.global_prefill_with_cache(d["q"], d["k"], d["v"], d["pos"], d["wq"], d["wk"], kc, vc, rotary_dim=R,
                                 theta=THETA, eps=EPS)
    st, detail = zg.device_status()
    assert st == -5 and (detail & 0xFF) == 4, (st, detail)
    assert zg.device_status()[0] == 0  # the record was cleared
    _check_slot(kc, vc, inp, 0, 2, 31, 31, "in range")


@pytest.mark.parametrize("D,HQ,HKV,R", [(128, 32, 8, 42), (64, 16, 8, 20)])
def test_prefill_then_decode_matches_the_longer_prefill(zg, D, HQ, HKV, R):
    # a two-layer stack (layer 0 local, layer 1 global): prefill L tokens with cache emission,
    # decode token L from those caches, and compare with the oracle's prefill of L + 1 tokens
    B, L, W, S = 2, 300, 128, 512
    layers = [_inputs(B, L + 1, seed=20 + l, d=D, Hq=HQ, Hkv=HKV) for l in range(2)]
    k_ring = torch.full((1, B, HKV, W, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    v_ring = k_ring.clone()
    k_glob = torch.full((1, B, HKV, S, D), SENTINEL, dtype=torch.bfloat16, device="cuda")
    v_glob = k_glob.clone()
    for l, inp in enumerate(layers):
        d = {k: v[:, :L].contiguous().cuda() if v.dim() > 1 else v.cuda() for k, v in inp.items()}
        if l == 0:
            zg.swa_prefill_with_cache(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], k_ring[0],
                                      v_ring[0], window=W, rotary_dim=R, theta=THETA, eps=EPS)
        else:
            zg.global_prefill_with_cache(d["q"], d["k"], d["v"], d["pos"], d["wq"], d["wk"], k_glob[0], v_glob[0],
                                         rotary_dim=R, theta=THETA, eps=EPS)
    step = {n: torch.stack([inp[n][:, L] for inp in layers]).contiguous().cuda() for n in ("q", "k", "v", "gate")}
    wq = torch.stack([inp["wq"] for inp in layers]).contiguous().cuda()
    wk = torch.stack([inp["wk"] for inp in layers]).contiguous().cuda()
    pos = layers[0]["pos"][:, L].contiguous().cuda()
    out = zg.hybrid_decode(step["q"], step["k"], step["v"], step["gate"], pos, wq, wk, [0, 1], k_glob, v_glob, k_ring,
                           v_ring, rotary_dim=R, theta=THETA, eps=EPS)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    for l, inp in enumerate(layers):
        rows = [b * (L + 1) + L for b in range(B)]
        ref = oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"] if l == 0 else None, inp["pos"],
                                  inp["wq"], inp["wk"], window=W if l == 0 else 0, rotary_dim=R, theta=THETA, eps=EPS,
                                  rows=rows)
        got = out[l].double().cpu().numpy().reshape(B, HQ, D)
        assert_close(got, ref.reshape(B, HQ, D), f"layer {l} decode after prefill")
