"""Decode over E4M3 (FP8) caches and the E4M3 cache writer: CUDA path through the C ABI.

The FP8 variant computes the decode step over the dequantised caches (stored / scale), so
the fp64 oracle is given exactly those values and the prefill's tolerance applies.  The
bytes the kernels store are checked against E4M3 rounding of the oracle's k_hat (within
half a unit in the last place: 2^-4 relative) and, for values, against torch's own
round-to-nearest conversion bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _case(NL, flags, B, Hq, Hkv, S, W, seed, k_scale, v_scale, d=128):
    g = torch.Generator().manual_seed(seed)
    NG, NS = sum(flags), NL - sum(flags)
    bf = lambda *sh: torch.randn(*sh, generator=g).bfloat16()
    inp = dict(q=bf(NL, B, Hq, d), k_new=bf(NL, B, Hkv, d), v_new=bf(NL, B, Hkv, d), gate=bf(NL, B, Hq, d),
               wq=0.5 + torch.rand(NL, d, generator=g), wk=0.5 + torch.rand(NL, d, generator=g))
    for name, shape, sc in (("k_glob", (NG, B, Hkv, S, d), k_scale), ("v_glob", (NG, B, Hkv, S, d), v_scale),
                            ("k_ring", (NS, B, Hkv, W, d), k_scale), ("v_ring", (NS, B, Hkv, W, d), v_scale)):
        inp[name] = workloads.to_e4m3(bf(*shape) * 2, sc)  # keys up to ~8: like RMS-normalised rows
    return inp


def _run(zg, inp, flags, positions, seqs, k_scale, v_scale, host=None, rotary_dim=42, theta=1e6, eps=1e-6):
    dev = {k: v.cuda() if v.device.type == "cpu" else v for k, v in inp.items()}
    if host is None:
        host = {k: inp[k][:, seqs].clone() for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    out = zg.hybrid_decode_fp8(dev["q"], dev["k_new"], dev["v_new"], dev["gate"], pos, dev["wq"], dev["wk"], flags,
                               dev["k_glob"], dev["v_glob"], dev["k_ring"], dev["v_ring"], k_scale=k_scale,
                               v_scale=v_scale, rotary_dim=rotary_dim, theta=theta, eps=eps)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    W = dev["k_ring"].shape[3]
    for si, b in enumerate(seqs):
        p = positions[b]
        # powers-of-two scales dequantise exactly in bf16 (half the host memory of the full-size case)
        exact_bf16 = all(float(np.log2(x)).is_integer() for x in (k_scale, v_scale))
        dt = torch.bfloat16 if exact_bf16 else torch.float64
        deq = {k: (host[k][:, si].to(dt) / (k_scale if k[0] == "k" else v_scale)) for k in host}
        ref, khat = oracle.decode_seq(inp["q"][:, b], inp["k_new"][:, b], inp["v_new"][:, b], inp["gate"][:, b],
                                      inp["wq"], inp["wk"], flags, deq["k_glob"], deq["v_glob"], deq["k_ring"],
                                      deq["v_ring"], p=p, rotary_dim=rotary_dim, theta=theta, eps=eps)
        assert_close(out[:, b].double().cpu().numpy(), ref, f"fp8 decode seq {b} p={p}")
        gi = ri = 0
        for l, f in enumerate(flags):
            kc, vc, slot = (dev["k_glob"][gi, b], dev["v_glob"][gi, b], p) if f else \
                (dev["k_ring"][ri, b], dev["v_ring"][ri, b], p % W)
            gi, ri = gi + (1 if f else 0), ri + (0 if f else 1)
            got_k = kc[:, slot].to(torch.float64).cpu().numpy()
            want_k = khat[l] * k_scale
            assert np.all(np.abs(got_k - want_k) <= 2.0 ** -4 * np.abs(want_k) + 2.0 ** -10), f"key slot layer {l}"
            want_v = (inp["v_new"][l, b].float() * v_scale).to(F8)
            assert torch.equal(vc[:, slot].cpu().view(torch.uint8), want_v.view(torch.uint8)), f"value slot layer {l}"


@pytest.mark.parametrize("d,Hq,Hkv", [(64, 8, 2), (128, 16, 1), (64, 12, 4), (128, 8, 8)])
def test_fp8_decode_head_sizes_and_gqa_ratios(zg, d, Hq, Hkv):
    flags = [1, 0, 0, 1]
    inp = _case(4, flags, 2, Hq, Hkv, 9000, 128, d + Hq, 1.0, 8.0, d=d)
    _run(zg, inp, flags, [8999, 77], [0, 1], 1.0, 8.0, rotary_dim=workloads.rotary_dim_for(d))


@pytest.mark.parametrize("positions,k_scale,v_scale", [([4999, 130, 50], 1.0, 8.0), ([0, 127, 4096], 2.0, 3.0),
                                                       ([4095, 126, 128], 0.5, 16.0)])
def test_small_fp8_decode(zg, positions, k_scale, v_scale):
    flags = [0, 0, 1, 0, 0, 1]
    inp = _case(6, flags, 3, 8, 2, 5000, 128, sum(positions), k_scale, v_scale)
    _run(zg, inp, flags, positions, [0, 1, 2], k_scale, v_scale)


def test_fp8_decode_only_local_and_only_global(zg):
    for flags in ([0, 0, 0], [1, 1]):
        inp = _case(len(flags), flags, 2, 4, 1, 300, 128, 11 + len(flags), 1.0, 8.0)
        _run(zg, inp, flags, [299, 10], [0, 1], 1.0, 8.0)


def test_fp8_cache_writer(zg):
    B, L, HQ, HKV, D, R, W, S = 2, 300, 32, 8, 128, 42, 128, 512
    g = torch.Generator().manual_seed(5)
    k = torch.randn(B, L, HKV, D, generator=g).bfloat16()
    v = torch.randn(B, L, HKV, D, generator=g).bfloat16()
    pos = torch.stack([torch.arange(L, dtype=torch.int32) + o for o in (0, 900)]).contiguous()
    wk = 0.5 + torch.rand(D, generator=g)
    ks, vs = 1.0, 8.0
    for ring, slots in ((True, W), (False, S)):
        if not ring:
            pos = torch.stack([torch.arange(L, dtype=torch.int32)] * B).contiguous()
        kc = torch.zeros(B, HKV, slots, D, dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        zg.kv_cache_write_fp8(k.cuda(), v.cuda(), pos.cuda(), wk.cuda(), kc, vc, ring=ring, k_scale=ks, v_scale=vs,
                              rotary_dim=R, theta=1e6)
        torch.cuda.synchronize()
        assert zg.device_status()[0] == 0
        for b in range(B):
            for i in (list(range(max(0, L - W), L, 17)) if ring else list(range(0, L, 29))) + [L - 1]:
                slot = int(pos[b, i]) % W if ring else int(pos[b, i])
                for gh in (0, 5):
                    x = k[b, i, gh].double().numpy()
                    want = oracle.rope(oracle.rmsnorm(x, wk.double().numpy(), 1e-6), R, int(pos[b, i]), 1e6) * ks
                    got = kc[b, gh, slot].cpu().view(F8).to(torch.float64).numpy()
                    assert np.all(np.abs(got - want) <= 2.0 ** -4 * np.abs(want) + 2.0 ** -10), (ring, b, i, gh)
                    want_v = (v[b, i, gh].float() * vs).to(F8).view(torch.uint8)
                    assert torch.equal(vc[b, gh, slot].cpu(), want_v), (ring, b, i, gh)


def test_full_fp8_decode_config(zg):
    """B=8, p=262143, 32 layers, 262144-position caches in E4M3 (scales 1 and 8, powers of two,
    so the dequantised host copies are exact in bf16).  Oracle on sequences 0 and 7."""
    c = workloads.HYBRID_DECODE
    tok = workloads.decode_token_inputs(c)
    bf = workloads.decode_caches_device(c, "cuda")
    f8 = {k: workloads.to_e4m3(v, 1.0 if k[0] == "k" else 8.0) for k, v in bf.items()}
    del bf
    seqs = [0, 7]
    host = {k: v[:, seqs].cpu() for k, v in f8.items()}
    inp = dict(tok, **f8)
    inp.pop("pos")
    inp.pop("is_global")
    _run(zg, inp, c.layer_flags(), [c.pos] * c.B, seqs, 1.0, 8.0, host=host, rotary_dim=c.rotary_dim,
         theta=c.theta, eps=c.eps)
