"""Gated sliding-window prefill on E4M3 (FP8) inputs and E4M3 tensor-core products, through the
C ABI, against the fp64 oracle fed the dequantised inputs (stored / scale, exact in fp64).

The path rounds q_hat, k_hat and the softmax weights P to E4M3 exactly as the E4M3 global
prefill does (the same kernel, with the window's key blocks and sigmoid(gate) in the epilogue),
so the tolerance derived there holds: rel-L2 <= 0.10 and max-abs <= 0.2 of the largest output.
The gate is bf16 and enters in fp32, so it adds nothing to that bound.
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
UNIT = dict(q=1.0, k=1.0, v=1.0)


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _inputs(B, L, Hq, Hkv, seed, scales, d=128, gate_mean=0.0):
    g = torch.Generator().manual_seed(seed)
    raw = dict(q=torch.randn(B, L, Hq, d, generator=g), k=torch.randn(B, L, Hkv, d, generator=g),
               v=torch.randn(B, L, Hkv, d, generator=g))
    stored = {n: workloads.to_e4m3(raw[n].bfloat16(), scales[n]).view(torch.uint8) for n in raw}
    deq = {n: stored[n].view(torch.float8_e4m3fn).double() / scales[n] for n in raw}
    gate = (torch.randn(B, L, Hq, d, generator=g) * 2.0 + gate_mean).bfloat16()
    extra = dict(gate=gate, pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
                 wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))
    return stored, deq, extra


def _run(zg, stored, extra, scales, window, rotary_dim=42, theta=1e4):
    dev = {k: v.cuda() for k, v in {**stored, **extra}.items()}
    out = zg.swa_prefill_fp8(dev["q"], dev["k"], dev["v"], dev["gate"], dev["pos"], dev["wq"], dev["wk"],
                             window=window, q_scale=scales["q"], k_scale=scales["k"], v_scale=scales["v"],
                             rotary_dim=rotary_dim, theta=theta)
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    assert st == 0, (st, hex(detail))
    return out


def _check(out, deq, extra, rows, window, what, rotary_dim=42, theta=1e4):
    ref = oracle.prefill_rows(deq["q"], deq["k"], deq["v"], extra["gate"].double(), extra["pos"], extra["wq"],
                              extra["wk"], window=window, rotary_dim=rotary_dim, theta=theta, eps=1e-6, rows=rows)
    got = rows_of(out, rows)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    bound = MAX_ABS_F8_FRAC * float(np.max(np.abs(ref)))
    print(f"{what}: rel_l2={rel:.4f} max_abs={max_abs:.4f} (bound {bound:.4f})")
    assert rel <= REL_L2_F8 and max_abs <= bound, f"{what}: max_abs={max_abs:.3e} (bound {bound:.3e}) rel_l2={rel:.3e}"


@pytest.mark.parametrize("B,L,Hq,Hkv,window", [
    (1, 1, 32, 8, 128),       # a single token
    (1, 300, 32, 8, 128),     # the ZGCM-1 local layer: several windows and a ragged tail
    (2, 129, 32, 8, 128),     # just past one window, two sequences
    (1, 600, 8, 8, 37),       # MHA, odd window: lower window edges inside key blocks
    (1, 500, 16, 2, 128),     # GQA 8:1
    (1, 450, 32, 2, 64),      # GQA 16:1, window 64
    (1, 257, 4, 2, 200),      # GQA 2:1, window wider than 128
    (1, 200, 32, 8, 1),       # window 1: each query sees only itself
    (2, 3000, 32, 8, 128),    # 752 work items: several per persistent CTA, every row checked
    (1, 5000, 8, 8, 200),     # MHA, up to four key blocks per item, 160 items (some CTAs take two)
    (2, 700, 12, 3, 128),     # three KV heads: no rotation shared across k_hat rows
    (2, 700, 16, 4, 96),      # four KV heads
])
def test_fp8_swa_all_rows(zg, B, L, Hq, Hkv, window):
    stored, deq, extra = _inputs(B, L, Hq, Hkv, seed=700 + L + window, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, window)
    _check(out, deq, extra, list(range(B * L)), window, f"fp8 swa B{B} L{L} {Hq}/{Hkv} W{window}")


@pytest.mark.parametrize("rot", [0, 64, 128])  # widths other than 42 take the general query transform
def test_fp8_swa_other_rotary_widths(zg, rot):
    stored, deq, extra = _inputs(2, 350, 32, 8, seed=800 + rot, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, 128, rotary_dim=rot)
    _check(out, deq, extra, list(range(2 * 350)), 128, f"fp8 swa rotary {rot}", rotary_dim=rot)


def test_fp8_swa_scales_and_suppressing_gate(zg):
    """Per-tensor scales other than one, and gate logits ~ N(-3, 2^2) (most outputs suppressed)."""
    sc = dict(q=3.0, k=0.37, v=12.5)
    stored, deq, extra = _inputs(2, 333, 32, 8, seed=71, scales=sc, gate_mean=-3.0)
    out = _run(zg, stored, extra, sc, 128)
    _check(out, deq, extra, list(range(2 * 333)), 128, "fp8 swa scaled, suppressing gate")


def test_fp8_swa_long_sequence_sampled_rows(zg):
    L = 8192
    stored, deq, extra = _inputs(1, L, 32, 8, seed=93, scales=UNIT)
    out = _run(zg, stored, extra, UNIT, 128)
    rows = sorted(set(workloads.edge_rows(L) + list(range(100, L, 613))))
    _check(out, deq, extra, rows, 128, "fp8 swa L8192")


def test_fp8_swa_close_to_bf16_path_and_deterministic(zg):
    stored, deq, extra = _inputs(2, 400, 32, 8, seed=9, scales=UNIT)
    a = _run(zg, stored, extra, UNIT, 128)
    b = _run(zg, stored, extra, UNIT, 128)
    assert torch.equal(a, b)
    dev = {n: deq[n].bfloat16().cuda() for n in ("q", "k", "v")}
    e = {k: v.cuda() for k, v in extra.items()}
    ref16 = zg.swa_prefill(dev["q"], dev["k"], dev["v"], e["gate"], e["pos"], e["wq"], e["wk"], window=128,
                           rotary_dim=42, theta=1e4)
    torch.cuda.synchronize()
    _, rel = errors(a.double().cpu().numpy(), ref16.double().cpu().numpy())
    assert rel <= REL_L2_F8, rel


def test_fp8_swa_rejects(zg):
    stored, _, extra = _inputs(1, 64, 8, 2, seed=1, scales=UNIT)
    dev = {k: v.cuda() for k, v in {**stored, **extra}.items()}
    with pytest.raises(zg.ZgError, match="ZG_ERR_SHAPE"):
        zg.swa_prefill_fp8(dev["q"], dev["k"], dev["v"], dev["gate"], dev["pos"], dev["wq"], dev["wk"], window=0,
                           rotary_dim=42, theta=1e4)
    with pytest.raises(zg.ZgError, match="ZG_ERR_SHAPE"):
        zg.swa_prefill_fp8(dev["q"], dev["k"], dev["v"], dev["gate"], dev["pos"], dev["wq"], dev["wk"], window=128,
                           v_scale=float("inf"), rotary_dim=42, theta=1e4)
