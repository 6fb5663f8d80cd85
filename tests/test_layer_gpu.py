"""A whole gated SWA layer from the hidden states, on the library's own tensor-core GEMM with the
fused epilogues (RMSNorm + RoPE of q and k from the fp32 accumulator, sigmoid of the gate) and the
attention on the pre-normalised tensors, against the fp64 oracle: numpy GEMMs around the C
oracle's attention.  Also the GEMM alone (zg_linear) against an fp64 matmul.

GEMM tolerance: bf16 inputs are exact in fp64; the kernel accumulates in fp32 and rounds the
output to bf16 (2^-9 relative), so rel-L2 <= 4e-3 and max-abs <= 8e-3 of the largest output
leave room for the fp32 sums while failing for any dropped or misplaced K block (errors of
order one)."""
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


@pytest.mark.parametrize("B,L,hidden,Hq,Hkv,d,window,rot", [
    (2, 300, 4096, 32, 8, 128, 128, 42),   # the ZGCM-1 local layer shape
    (1, 200, 512, 4, 1, 128, 128, 42),     # GQA 4, small hidden
    (1, 333, 520, 8, 4, 64, 77, 20),       # d = 64, GQA 2, hidden not a multiple of 64, odd window
    (2, 150, 1024, 16, 2, 128, 128, 64),   # GQA 8, rotary_dim 64
    (1, 160, 768, 32, 2, 64, 50, 0),       # GQA 16, no rotation
])
def test_gated_swa_layer_matches_the_oracle(zg, B, L, hidden, Hq, Hkv, d, window, rot):
    inp = _layer_inputs(B, L, hidden, Hq, Hkv, d, seed=hidden + L)
    dv = {k: v.cuda() for k, v in inp.items()}
    y = zg.gated_swa_layer(dv["h"], dv["w_q"], dv["w_k"], dv["w_v"], dv["w_g"], dv["w_o"], dv["pos"], dv["wq"],
                           dv["wk"], Hq=Hq, Hkv=Hkv, window=window, rotary_dim=rot, theta=1e4)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    ref = _oracle_layer(inp, Hq, Hkv, d, window, rot, 1e4, 1e-6)
    assert_close(y.double().cpu().numpy(), ref, f"layer B{B} L{L} hidden {hidden} {Hq}/{Hkv} d{d}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (300, 264, 200), (128, 256, 64), (1000, 1032, 1000),
                                   (4096, 4096, 4096)])
def test_linear_matches_an_fp64_matmul(zg, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    x = torch.randn(M, K, generator=g).bfloat16()
    w = (torch.randn(K, N, generator=g) / K ** 0.5).bfloat16()
    y = zg.linear(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    rows = np.arange(M) if M <= 1000 else np.random.default_rng(0).choice(M, 300, replace=False)
    ref = x.double().numpy()[rows] @ w.double().numpy()
    got = y.double().cpu().numpy()[rows]
    err = np.abs(got - ref)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= 4e-3 and err.max() <= 8e-3 * np.abs(ref).max(), (rel, err.max(), np.abs(ref).max())


def test_gated_swa_layer_is_deterministic(zg):
    inp = {k: v.cuda() for k, v in _layer_inputs(1, 256, 1024, 8, 2, 128, seed=5).items()}
    run = lambda: zg.gated_swa_layer(inp["h"], inp["w_q"], inp["w_k"], inp["w_v"], inp["w_g"], inp["w_o"], inp["pos"],
                                     inp["wq"], inp["wk"], Hq=8, Hkv=2, rotary_dim=42, theta=1e4)
    assert torch.equal(run(), run())
