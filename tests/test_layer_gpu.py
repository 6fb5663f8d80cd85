"""A whole gated SWA layer from the hidden states (projections on cuBLASLt around the
library's attention) against the fp64 oracle: numpy GEMMs around the C oracle's attention."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _layer_inputs(B, L, hidden, Hq, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    w = lambda n_in, n_out: (torch.randn(n_in, n_out, generator=g) / n_in ** 0.5).bfloat16()
    return dict(h=torch.randn(B, L, hidden, generator=g).bfloat16(), w_q=w(hidden, Hq * d), w_k=w(hidden, Hkv * d),
                w_v=w(hidden, Hkv * d), w_g=w(hidden, Hq * d), w_o=w(Hq * d, hidden),
                pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
                wq=0.5 + torch.rand(d, generator=g), wk=0.5 + torch.rand(d, generator=g))


def _oracle_layer(inp, Hq, Hkv, d, window, rotary_dim, theta, eps):
    h = inp["h"].double().numpy()
    B, L, hidden = h.shape
    x = h.reshape(B * L, hidden)
    proj = lambda w, heads: (x @ inp[w].double().numpy()).reshape(B, L, heads, d)
    q, k, v, gate = proj("w_q", Hq), proj("w_k", Hkv), proj("w_v", Hkv), proj("w_g", Hq)
    a = oracle.prefill_rows(q, k, v, gate, inp["pos"], inp["wq"], inp["wk"], window=window, rotary_dim=rotary_dim,
                            theta=theta, eps=eps, rows=list(range(B * L)))
    return (a.reshape(B * L, Hq * d) @ inp["w_o"].double().numpy()).reshape(B, L, hidden)


@pytest.mark.parametrize("B,L,hidden,Hq,Hkv,d", [(2, 300, 4096, 32, 8, 128), (1, 200, 512, 4, 1, 128)])
def test_gated_swa_layer_matches_the_oracle(zg, B, L, hidden, Hq, Hkv, d):
    inp = _layer_inputs(B, L, hidden, Hq, Hkv, d, seed=hidden + L)
    dv = {k: v.cuda() for k, v in inp.items()}
    y = zg.gated_swa_layer(dv["h"], dv["w_q"], dv["w_k"], dv["w_v"], dv["w_g"], dv["w_o"], dv["pos"], dv["wq"],
                           dv["wk"], Hq=Hq, Hkv=Hkv, window=128, rotary_dim=42, theta=1e4)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    ref = _oracle_layer(inp, Hq, Hkv, d, 128, 42, 1e4, 1e-6)
    assert_close(y.double().cpu().numpy(), ref, f"layer B{B} L{L} hidden {hidden}")


def test_gated_swa_layer_is_deterministic(zg):
    inp = {k: v.cuda() for k, v in _layer_inputs(1, 256, 1024, 8, 2, 128, seed=5).items()}
    run = lambda: zg.gated_swa_layer(inp["h"], inp["w_q"], inp["w_k"], inp["w_v"], inp["w_g"], inp["w_o"], inp["pos"],
                                     inp["wq"], inp["wk"], Hq=8, Hkv=2, rotary_dim=42, theta=1e4)
    assert torch.equal(run(), run())
