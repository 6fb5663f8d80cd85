"""Global prefill on E4M3 (FP8) inputs and E4M3 tensor-core products, through the C ABI.

The oracle is given the dequantised inputs (stored / scale, exact in fp64), so what remains
is the rounding of the path itself: q_hat and k_hat to E4M3 (3 mantissa bits, relative
rounding error up to 2^-4, about 2^-4/sqrt(3) = 3.6% rms) and the softmax weights P to E4M3
(the same).  A score s = q_hat.k_hat/sqrt(d) with both factors so rounded carries an error
of about sqrt(2) x 3.6% of the rms score term (~5%), which moves each softmax weight by
~5% relatively; P's own rounding adds ~3.6%; the two are independent, so the output's
relative L2 error is about sqrt(0.05^2 + 0.036^2) = 6%.  The tests bound it by 0.10 and the
largest element error by 0.2 of the largest output magnitude (4 to 5 standard deviations of
the element error over ~1e5 elements); the bf16 path's bounds (1e-2) do not apply here.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import errors, rows_of

pytestmark = pytest.mark.gpu

REL_L2_F8 = 0.10
MAX_ABS_F8_FRAC = 0.2


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _inputs(B, L, Hq, Hkv, d, seed, scales, spread=1.0):
    g = torch.Generator().manual_seed(seed)
    raw = dict(q=torch.randn(B, L, Hq, d, generator=g) * spread, k=torch.randn(B, L, Hkv, d, generator=g) * spread,
               v=torch.randn(B, L, Hkv, d, generator=g))
    stored = {n: workloads.to_e4m3(raw[n].bfloat16(), scales[n]).view(torch.uint8) for n in raw}
    deq = {n: stored[n].view(torch.float8_e4m3fn).double() / scales[n] for n in raw}
    extra = dict(pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
                 wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))
    return stored, deq, extra


def _run(zg, stored, extra, scales, rotary_dim, theta, eps=1e-6):
    dev = {k: v.cuda() for k, v in {**stored, **extra}.items()}
    out = zg.global_prefill_fp8(dev["q"], dev["k"], dev["v"], dev["pos"], dev["wq"], dev["wk"],
                                q_scale=scales["q"], k_scale=scales["k"], v_scale=scales["v"], rotary_dim=rotary_dim,
                                theta=theta, eps=eps)
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    assert st == 0, (st, hex(detail))
    return out


def _check(out, deq, extra, rows, rotary_dim, theta, what, eps=1e-6):
    ref = oracle.prefill_rows(deq["q"], deq["k"], deq["v"], None, extra["pos"], extra["wq"], extra["wk"], window=0,
                              rotary_dim=rotary_dim, theta=theta, eps=eps, rows=rows)
    got = rows_of(out, rows)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    bound = MAX_ABS_F8_FRAC * float(np.max(np.abs(ref)))
    print(f"{what}: rel_l2={rel:.4f} max_abs={max_abs:.4f} (bound {bound:.4f})")
    assert rel <= REL_L2_F8 and max_abs <= bound, f"{what}: max_abs={max_abs:.3e} (bound {bound:.3e}) rel_l2={rel:.3e}"
    return rel


UNIT = dict(q=1.0, k=1.0, v=1.0)


@pytest.mark.parametrize("B,L", [(1, 1), (1, 31), (2, 129), (2, 300), (1, 1000)])
def test_fp8_small_lengths_all_rows(zg, B, L):
    stored, deq, extra = _inputs(B, L, 32, 8, 128, seed=500 + L + B, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, 42, 1e6)
    _check(out, deq, extra, list(range(B * L)), 42, 1e6, f"fp8 global B{B} L{L}")


@pytest.mark.parametrize("rot", [64, 42])  # the general query transform, and the one with 42 compiled in
@pytest.mark.parametrize("Hq,Hkv,L", [(8, 8, 600), (4, 2, 530), (16, 2, 450), (32, 2, 300)])
def test_fp8_gqa_ratios(zg, Hq, Hkv, L, rot):
    stored, deq, extra = _inputs(1, L, Hq, Hkv, 128, seed=Hq * 7 + Hkv, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, rot, 1e4)
    _check(out, deq, extra, list(range(L)), rot, 1e4, f"fp8 global {Hq}/{Hkv} L{L} rotary {rot}")


@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (12, 3)])  # KV heads per token not a multiple of 8
def test_fp8_kv_head_counts(zg, Hq, Hkv):
    """The k_hat pre-pass shares each token's rotation among its consecutive KV-head rows (4 lanes
    here, or none for 3 heads); the whole output against the oracle."""
    stored, deq, extra = _inputs(2, 333, Hq, Hkv, 128, seed=40 + Hkv, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, 42, 1e6)
    _check(out, deq, extra, list(range(2 * 333)), 42, 1e6, f"fp8 global {Hq}/{Hkv}")


def test_fp8_scales_other_than_one(zg):
    """Per-tensor scales (not powers of two) are divided out: the same attention as unit scales
    of the same dequantised values, within the tolerance."""
    sc = dict(q=3.0, k=0.37, v=12.5)
    stored, deq, extra = _inputs(2, 257, 32, 8, 128, seed=77, scales=sc, spread=2.0)
    out = _run(zg, stored, extra, sc, 42, 1e6)
    _check(out, deq, extra, list(range(2 * 257)), 42, 1e6, "fp8 global scaled")


def test_fp8_long_sequence_sampled_rows(zg):
    """8K tokens: 64 key blocks per row at the end, the running maximum raised many times."""
    L = 8192
    stored, deq, extra = _inputs(1, L, 32, 8, 128, seed=91, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, 42, 1e6)
    rows = workloads.edge_rows(L) + list(range(1000, L, 997))
    _check(out, deq, extra, sorted(set(rows)), 42, 1e6, "fp8 global L8192")


def test_fp8_peaked_scores(zg):
    """Larger inputs (scores spread over tens of units): the softmax is dominated by a few keys,
    the regime where the E4M3 weights' relative rounding is felt most."""
    stored, deq, extra = _inputs(1, 700, 32, 8, 128, seed=13, scales=dict(q=1.0, k=1.0, v=1.0), spread=1.0)
    extra["wq"] = extra["wq"] * 2.0
    extra["wk"] = extra["wk"] * 2.0
    out = _run(zg, stored, extra, UNIT, 42, 1e6)
    _check(out, deq, extra, list(range(700)), 42, 1e6, "fp8 global peaked")


def test_fp8_deterministic_and_close_to_bf16_path(zg):
    """Two runs give the same bytes; the bf16 path over the same dequantised inputs (exact in
    bf16 for unit scales) agrees with it within the E4M3 tolerance."""
    stored, deq, extra = _inputs(2, 400, 32, 8, 128, seed=5, scales=UNIT)
    a = _run(zg, stored, extra, UNIT, 42, 1e6)
    b = _run(zg, stored, extra, UNIT, 42, 1e6)
    assert torch.equal(a, b)
    dev = {n: deq[n].bfloat16().cuda() for n in ("q", "k", "v")}
    e = {k: v.cuda() for k, v in extra.items()}
    ref16 = zg.global_prefill(dev["q"], dev["k"], dev["v"], e["pos"], e["wq"], e["wk"], rotary_dim=42, theta=1e6)
    torch.cuda.synchronize()
    _, rel = errors(a.double().cpu().numpy(), ref16.double().cpu().numpy())
    assert rel <= REL_L2_F8, rel


def test_fp8_rejects(zg):
    stored, _, extra = _inputs(1, 64, 8, 2, 128, seed=1, scales=UNIT)
    dev = {k: v.cuda() for k, v in {**stored, **extra}.items()}
    with pytest.raises(zg.ZgError, match="ZG_ERR_SHAPE"):
        zg.global_prefill_fp8(dev["q"], dev["k"], dev["v"], dev["pos"], dev["wq"], dev["wk"], k_scale=0.0,
                              rotary_dim=42, theta=1e6)
    q64 = torch.zeros(1, 64, 8, 64, dtype=torch.uint8, device="cuda")
    k64 = torch.zeros(1, 64, 2, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(zg.ZgError, match="ZG_ERR_UNSUPPORTED"):
        zg.global_prefill_fp8(q64, k64, k64, dev["pos"], dev["wq"][:64].contiguous(), dev["wk"][:64].contiguous(),
                              rotary_dim=32, theta=1e6)
    q3 = torch.zeros(1, 64, 6, 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(zg.ZgError, match="ZG_ERR_UNSUPPORTED"):
        zg.global_prefill_fp8(q3, dev["k"], dev["v"], dev["pos"], dev["wq"], dev["wk"], rotary_dim=42, theta=1e6)
