"""Pins for the backward oracle (oracle/backward.py), CPU only: its fp64 forward agrees
with the independent C oracle, autograd agrees with central finite differences, and
the window-1 case reduces to closed forms."""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bw


def _small(B=1, L=9, Hq=4, Hkv=2, d=16, seed=0):
    g = torch.Generator().manual_seed(seed)
    return dict(q=torch.randn(B, L, Hq, d, generator=g, dtype=torch.float64),
                k=torch.randn(B, L, Hkv, d, generator=g, dtype=torch.float64),
                v=torch.randn(B, L, Hkv, d, generator=g, dtype=torch.float64),
                gate=torch.randn(B, L, Hq, d, generator=g, dtype=torch.float64),
                pos=(torch.arange(L, dtype=torch.int32) + 3).repeat(B, 1),
                # norm weights are fp32 in the interface: draw them exactly representable there
                wq=(0.5 + torch.rand(d, generator=g)).double(),
                wk=(0.5 + torch.rand(d, generator=g)).double(),
                dout=torch.randn(B, L, Hq, d, generator=g, dtype=torch.float64))


@pytest.mark.parametrize("window,gated", [(4, True), (0, False)])
def test_forward_agrees_with_the_c_oracle(window, gated):
    x = _small(B=2, L=12, Hq=4, Hkv=1, d=16, seed=1)
    gate = x["gate"] if gated else None
    out = bw.forward(x["q"], x["k"], x["v"], gate, x["pos"], x["wq"], x["wk"], window=window, rotary_dim=6,
                     theta=1e4, eps=1e-6).numpy()
    ref = oracle.prefill_rows(x["q"], x["k"], x["v"], gate, x["pos"], x["wq"], x["wk"], window=window, rotary_dim=6,
                              theta=1e4, eps=1e-6, rows=list(range(24)))
    assert np.abs(out.reshape(24, 4, 16) - ref).max() < 1e-12


@pytest.mark.parametrize("window,gated", [(4, True), (0, False)])
def test_gradients_agree_with_finite_differences(window, gated):
    x = _small(seed=2)
    gate = x["gate"] if gated else None
    kw = dict(window=window, rotary_dim=6, theta=1e4, eps=1e-6)
    grads = bw.gradients(x["q"], x["k"], x["v"], gate, x["pos"], x["wq"], x["wk"], x["dout"], **kw)

    def loss(name, idx, delta):
        t = {n: (x[n].clone() if x[n] is not None else None) for n in ("q", "k", "v", "gate")}
        t[name][idx] += delta
        o = bw.forward(t["q"], t["k"], t["v"], t["gate"] if gated else None, x["pos"], x["wq"], x["wk"], **kw)
        return float((o * x["dout"]).sum())

    rng = np.random.default_rng(3)
    for name, gi in (("q", 0), ("k", 1), ("v", 2), ("gate", 3)):
        if name == "gate" and not gated:
            assert grads[3] is None
            continue
        shape = x[name].shape
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in shape)
            h = 1e-5
            fd = (loss(name, idx, h) - loss(name, idx, -h)) / (2 * h)
            an = float(grads[gi][idx])
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


def test_window_one_closed_forms():
    # each token attends only to itself: out = v * sigmoid(g), so dv_j = sum over the G query heads of
    # dout * sigmoid(g), dgate = dout * v * sigmoid'(g), and dq = dk = 0
    x = _small(B=1, L=5, Hq=4, Hkv=2, d=8, seed=4)
    dq, dk, dv, dg = bw.gradients(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], x["dout"],
                                  window=1, rotary_dim=4, theta=1e4, eps=1e-6)
    sg = torch.sigmoid(x["gate"])
    vv = x["v"].repeat_interleave(2, dim=2)
    assert torch.allclose(dg, x["dout"] * vv * sg * (1 - sg), atol=1e-12)
    assert torch.allclose(dv, (x["dout"] * sg).reshape(1, 5, 2, 2, 8).sum(dim=3), atol=1e-12)
    assert float(dq.abs().max()) < 1e-12 and float(dk.abs().max()) < 1e-12
