"""Gated sliding-window prefill: CUDA path (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, rows_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _run(zg, inp, window, rotary_dim, theta, eps=1e-6):
    d = _to_dev(inp)
    out = zg.swa_prefill(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], window=window,
                         rotary_dim=rotary_dim, theta=theta, eps=eps)
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    assert st == 0, (st, detail)
    return out


def _check(zg, inp, rows, window, rotary_dim, theta, what, eps=1e-6):
    out = _run(zg, inp, window, rotary_dim, theta, eps)
    ref = oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"], inp["pos"], inp["wq"], inp["wk"],
                              window=window, rotary_dim=rotary_dim, theta=theta, eps=eps, rows=rows)
    return assert_close(rows_of(out, rows), ref, what), out


def _synthetic(B, L, Hq, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return dict(q=torch.randn(B, L, Hq, d, generator=g).bfloat16(), k=torch.randn(B, L, Hkv, d, generator=g).bfloat16(),
                v=torch.randn(B, L, Hkv, d, generator=g).bfloat16(), gate=torch.randn(B, L, Hq, d, generator=g).bfloat16(),
                pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
                wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))


def test_tiny_config_all_rows(zg):
    c = workloads.TINY_SWA
    inp = workloads.prefill_inputs(c)
    _check(zg, inp, workloads.sample_rows(c), c.window, c.rotary_dim, c.theta, c.name)


@pytest.mark.parametrize("B,L,Hq,Hkv,d,window", [
    (1, 1, 4, 1, 64, 128),      # single token
    (2, 33, 4, 1, 64, 128),     # one full tile + 1 (ragged tail)
    (1, 127, 32, 8, 128, 128),  # just under the window
    (1, 129, 32, 8, 128, 128),  # just over the window
    (2, 300, 32, 8, 128, 128),  # several tiles, ragged
    (1, 200, 4, 1, 128, 1),     # window 1: out = v * sigmoid(g)
    (1, 170, 8, 2, 64, 37),     # odd window
    (1, 150, 8, 1, 128, 128),   # GQA 8:1 (16 tokens per tile)
    (1, 150, 4, 2, 128, 128),   # GQA 2:1
    (1, 150, 2, 2, 64, 128),    # MHA (128 tokens per tile)
    (2, 170, 32, 2, 128, 128),  # GQA 16:1 (8 tokens per tile)
    (1, 140, 16, 1, 64, 100),   # GQA 16:1, d = 64
])
def test_edge_shapes(zg, B, L, Hq, Hkv, d, window):
    inp = _synthetic(B, L, Hq, Hkv, d, seed=B * 1000 + L + d + window)
    r = workloads.rotary_dim_for(d)
    _check(zg, inp, list(range(B * L)), window, r, 1e4, f"B{B} L{L} {Hq}/{Hkv} d{d} W{window}")


def test_rotary_dim_zero_and_full(zg):
    inp = _synthetic(1, 160, 4, 1, 64, seed=5)
    _check(zg, inp, list(range(160)), 128, 0, 1e4, "r=0")
    _check(zg, inp, list(range(160)), 128, 64, 1e4, "r=d")


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (8, 1, 128), (4, 2, 64)])
def test_large_weights_take_exact_maximum(zg, Hq, Hkv, d):
    # RMSNorm weights of magnitude ~3-4.5 put the score bound sqrt(d) max|wq| * sqrt(d) max|wk|
    # far above 50 log2 units, so the softmax takes the two-pass row maximum instead of the bound
    inp = _synthetic(1, 300, Hq, Hkv, d, seed=77 + d + Hq)
    inp["wq"] = inp["wq"] * 3.0
    inp["wk"] = inp["wk"] * 3.0
    _check(zg, inp, list(range(300)), 128, workloads.rotary_dim_for(d), 1e4, f"large weights {Hq}/{Hkv} d{d}")


def test_swa_4k_config(zg):
    c = workloads.SWA_4K
    inp = workloads.prefill_inputs(c)
    _check(zg, inp, workloads.sample_rows(c), c.window, c.rotary_dim, c.theta, c.name)


def test_swa_256k_outlier_config(zg):
    c = workloads.SWA_256K
    inp = workloads.prefill_inputs(c)
    _check(zg, inp, workloads.sample_rows(c), c.window, c.rotary_dim, c.theta, c.name)


def test_deterministic_and_position_shift(zg):
    inp = _synthetic(1, 400, 32, 8, 128, seed=9)
    a = _run(zg, inp, 128, 42, 1e6)
    b = _run(zg, inp, 128, 42, 1e6)
    assert torch.equal(a, b)
    shifted = dict(inp, pos=inp["pos"] + 200000)
    c = _run(zg, shifted, 128, 42, 1e6)
    assert_close(c.double().cpu().numpy(), a.double().cpu().numpy(), "position shift")


def test_bounded_wait_times_out_and_context_survives(zg):
    zg.device_status()
    zg.selftest_bounded_wait(2_000_000)  # 2 ms
    st, detail = zg.device_status()
    assert st == -8 and (detail >> 8) == 99 and (detail & 0xFF) == 1
    assert zg.device_status()[0] == 0  # cleared
    # the context is still usable
    inp = _synthetic(1, 40, 4, 1, 64, seed=3)
    _check(zg, inp, list(range(40)), 128, 20, 1e4, "after timeout")
