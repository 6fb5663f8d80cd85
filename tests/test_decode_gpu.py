"""Hybrid decode step: CUDA path (through the C ABI) against the fp64 oracle, per sequence."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _draw(shape, g):
    return torch.randn(*shape, generator=g).bfloat16()


def _small_case(NL, flags, B, Hq, Hkv, S, W, seed, d=128):
    g = torch.Generator().manual_seed(seed)
    NG = sum(flags)
    NS = NL - NG
    return dict(q=_draw((NL, B, Hq, d), g), k_new=_draw((NL, B, Hkv, d), g), v_new=_draw((NL, B, Hkv, d), g),
                gate=_draw((NL, B, Hq, d), g), wq=0.5 + torch.rand(NL, d, generator=g),
                wk=0.5 + torch.rand(NL, d, generator=g),
                k_glob=_draw((NG, B, Hkv, S, d), g), v_glob=_draw((NG, B, Hkv, S, d), g),
                k_ring=_draw((NS, B, Hkv, W, d), g), v_ring=_draw((NS, B, Hkv, W, d), g))


def _run_and_check(zg, inp, flags, positions, rotary_dim, theta, eps, seqs, host_caches=None):
    """inp: tensors (host or device).  host_caches: pre-step host copies of the caches for `seqs`
    (dict of [N*, len(seqs), ...]) when the device caches were drawn on the device."""
    dev = {k: v.cuda() if v.device.type == "cpu" else v for k, v in inp.items()}
    if host_caches is None:
        host_caches = {k: inp[k][:, seqs].clone() for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    out = zg.hybrid_decode(dev["q"], dev["k_new"], dev["v_new"], dev["gate"], pos, dev["wq"], dev["wk"], flags,
                           dev["k_glob"], dev["v_glob"], dev["k_ring"], dev["v_ring"], rotary_dim=rotary_dim,
                           theta=theta, eps=eps)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    W = dev["k_ring"].shape[3]
    results = []
    for si, b in enumerate(seqs):
        p = positions[b]
        ref, khat = oracle.decode_seq(inp["q"][:, b].cpu(), inp["k_new"][:, b].cpu(), inp["v_new"][:, b].cpu(),
                                      inp["gate"][:, b].cpu(), inp["wq"].cpu(), inp["wk"].cpu(), flags,
                                      host_caches["k_glob"][:, si], host_caches["v_glob"][:, si],
                                      host_caches["k_ring"][:, si], host_caches["v_ring"][:, si],
                                      p=p, rotary_dim=rotary_dim, theta=theta, eps=eps)
        results.append(assert_close(out[:, b].double().cpu().numpy(), ref, f"decode seq {b} p={p}"))
        # the cache slot written for the new token
        gi = si_ = 0
        for l, f in enumerate(flags):
            if f:
                kk = dev["k_glob"][gi, b, :, p].double().cpu().numpy()
                vv = dev["v_glob"][gi, b, :, p]
                gi += 1
            else:
                kk = dev["k_ring"][si_, b, :, p % W].double().cpu().numpy()
                vv = dev["v_ring"][si_, b, :, p % W]
                si_ += 1
            assert_close(kk, khat[l], f"cache key layer {l}")
            assert torch.equal(vv.cpu(), inp["v_new"][l, b].cpu())
    return out, results


@pytest.mark.parametrize("positions", [[4999, 130, 50], [0, 127, 4096], [4095, 126, 128]])
def test_small_hybrid_decode(zg, positions):
    flags = [0, 0, 1, 0, 0, 1]
    inp = _small_case(6, flags, 3, 8, 2, 5000, 128, seed=sum(positions))
    _run_and_check(zg, inp, flags, positions, 42, 1e6, 1e-6, seqs=[0, 1, 2])


@pytest.mark.parametrize("d,Hq,Hkv,W", [
    (64, 8, 8, 128),     # no head sharing, d = 64
    (64, 8, 4, 128),     # GQA 2:1
    (128, 16, 2, 128),   # GQA 8:1
    (128, 32, 2, 128),   # GQA 16:1 (two groups of 8 fragment rows)
    (64, 16, 1, 128),    # GQA 16:1, d = 64
    (128, 12, 4, 128),   # GQA 3:1 (not a power of two)
    (128, 8, 2, 200),    # a 200-slot ring (stages past the ring read as zeros)
    (64, 8, 2, 40),      # a 40-slot ring
])
def test_decode_head_sizes_gqa_ratios_and_windows(zg, d, Hq, Hkv, W):
    flags = [0, 1, 0, 1]
    S = 9000  # two splits of 8192 keys
    inp = _small_case(len(flags), flags, 3, Hq, Hkv, S, W, seed=d + Hq + W, d=d)
    positions = [8999, 8192, min(W, 30)]
    _run_and_check(zg, inp, flags, positions, workloads.rotary_dim_for(d), 1e6, 1e-6, seqs=[0, 1, 2])


def test_decode_only_local_and_only_global(zg):
    for flags in ([0, 0, 0], [1, 1]):
        inp = _small_case(len(flags), flags, 2, 4, 1, 300, 128, seed=7 + len(flags))
        _run_and_check(zg, inp, flags, [299, 10], 42, 1e6, 1e-6, seqs=[0, 1])


def test_decode_position_outside_cache_is_inert(zg):
    flags = [0, 1]
    inp = _small_case(2, flags, 1, 4, 1, 300, 128, seed=3)
    dev = {k: v.cuda() for k, v in inp.items()}
    before = {k: dev[k].clone() for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
    pos = torch.tensor([300], dtype=torch.int32, device="cuda")
    out = zg.hybrid_decode(dev["q"], dev["k_new"], dev["v_new"], dev["gate"], pos, dev["wq"], dev["wk"], flags,
                           dev["k_glob"], dev["v_glob"], dev["k_ring"], dev["v_ring"], rotary_dim=42, theta=1e6)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    for k in before:
        assert torch.equal(before[k], dev[k])


def test_full_hybrid_decode_config(zg):
    """B=8, p=262143, 32 layers (global at 5,11,17,23,29), caches of 262144 positions.
    Oracle on sequences 0 and 7 (every layer), from host copies taken before the step."""
    c = workloads.HYBRID_DECODE
    tok = workloads.decode_token_inputs(c)
    caches = workloads.decode_caches_device(c, "cuda")
    seqs = [0, 7]
    host = {k: v[:, seqs].cpu() for k, v in caches.items()}
    inp = dict(tok, **caches)
    inp.pop("pos")
    inp.pop("is_global")
    flags = c.layer_flags()
    _run_and_check(zg, inp, flags, [c.pos] * c.B, c.rotary_dim, c.theta, c.eps, seqs=seqs, host_caches=host)


def test_two_chained_steps_see_the_written_slot(zg):
    """Step at p, then at p + 1 on the same device caches: the second step must attend to the key and
    value the first one wrote (and, at p + 1 = 128, a ring must have dropped position 0).  The oracle's
    caches for the second step are the pre-step caches with slot p holding the oracle's own k_hat of
    step 1 (in the bf16 cache format) and step 1's v_new."""
    flags = [0, 1, 0, 0, 1]
    NL, B, Hq, Hkv, S, W = len(flags), 2, 8, 2, 600, 128
    first = _small_case(NL, flags, B, Hq, Hkv, S, W, seed=31)
    g = torch.Generator().manual_seed(32)
    second = {k: _draw(tuple(first[k].shape), g) for k in ("q", "k_new", "v_new", "gate")}
    positions = [127, 598]
    dev = {k: v.cuda() for k, v in first.items()}
    pre = {k: first[k].clone() for k in ("k_glob", "v_glob", "k_ring", "v_ring")}
    outs = []
    for step, x in enumerate((first, second)):
        pos = torch.tensor([p + step for p in positions], dtype=torch.int32, device="cuda")
        xd = {k: x[k].cuda() for k in ("q", "k_new", "v_new", "gate")}
        outs.append(zg.hybrid_decode(xd["q"], xd["k_new"], xd["v_new"], xd["gate"], pos, dev["wq"], dev["wk"], flags,
                                     dev["k_glob"], dev["v_glob"], dev["k_ring"], dev["v_ring"], rotary_dim=42,
                                     theta=1e6))
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    for b, p in enumerate(positions):
        args = dict(rotary_dim=42, theta=1e6, eps=1e-6)
        caches = {k: pre[k][:, b].clone() for k in pre}
        _, khat = oracle.decode_seq(first["q"][:, b], first["k_new"][:, b], first["v_new"][:, b],
                                    first["gate"][:, b], first["wq"], first["wk"], flags, caches["k_glob"],
                                    caches["v_glob"], caches["k_ring"], caches["v_ring"], p=p, **args)
        gi = si = 0
        for l, f in enumerate(flags):
            kk = torch.from_numpy(khat[l]).to(torch.bfloat16)
            if f:
                caches["k_glob"][gi, :, p] = kk
                caches["v_glob"][gi, :, p] = first["v_new"][l, b]
                gi += 1
            else:
                caches["k_ring"][si, :, p % W] = kk
                caches["v_ring"][si, :, p % W] = first["v_new"][l, b]
                si += 1
        ref2, _ = oracle.decode_seq(second["q"][:, b], second["k_new"][:, b], second["v_new"][:, b],
                                    second["gate"][:, b], first["wq"], first["wk"], flags, caches["k_glob"],
                                    caches["v_glob"], caches["k_ring"], caches["v_ring"], p=p + 1, **args)
        assert_close(outs[1][:, b].double().cpu().numpy(), ref2, f"second step seq {b} p={p + 1}")
