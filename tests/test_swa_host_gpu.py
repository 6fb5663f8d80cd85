"""The gated SWA prefill from host buffers (zg_swa_prefill_host): chunked, with the copies inside
the call, against the fp64 oracle and against the device-buffer call on the same inputs.

Each chunk carries the window's key halo, so every output row sees exactly the keys of one
whole-sequence call; only the order in which a tile's keys sit in the kernel's key ring can
differ, which moves fp32 sums by rounding, so the comparison with the device-buffer call is
rel-L2 <= 1e-3 (bf16 outputs: a few units in the last place at most) and the oracle
comparison uses the prefill's own bars.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_close, errors, rows_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _inputs(B, L, Hq, Hkv, seed, pin=True):
    g = torch.Generator().manual_seed(seed)
    x = dict(q=torch.randn(B, L, Hq, 128, generator=g).bfloat16(), k=torch.randn(B, L, Hkv, 128, generator=g).bfloat16(),
             v=torch.randn(B, L, Hkv, 128, generator=g).bfloat16(),
             gate=torch.randn(B, L, Hq, 128, generator=g).bfloat16(),
             pos=torch.arange(L, dtype=torch.int32).repeat(B, 1).contiguous(),
             wq=0.5 + torch.rand(128, generator=g), wk=0.5 + torch.rand(128, generator=g))
    return {k: (v.pin_memory() if pin else v) for k, v in x.items()}


def _device_call(zg, x, window):
    d = {k: v.cuda() for k, v in x.items()}
    out = zg.swa_prefill(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], window=window,
                         rotary_dim=42, theta=1e4)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("B,L,Hq,Hkv,window,chunk", [
    (2, 1000, 32, 8, 128, 256),   # four chunks, the last one ragged
    (1, 777, 32, 8, 37, 300),     # odd window (halo rounded up to 128), chunks not multiples of the tile
    (1, 300, 16, 2, 128, 1024),   # one chunk longer than the sequence; GQA 8
])
def test_host_call_matches_oracle_and_device_call(zg, B, L, Hq, Hkv, window, chunk):
    x = _inputs(B, L, Hq, Hkv, seed=L + chunk)
    out = zg.swa_prefill_host(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=window,
                              rotary_dim=42, theta=1e4, chunk_tokens=chunk)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    assert not out.is_cuda
    rows = list(range(B * L))
    ref = oracle.prefill_rows(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=window,
                              rotary_dim=42, theta=1e4, eps=1e-6, rows=rows)
    assert_close(rows_of(out, rows), ref, f"host call B{B} L{L} W{window} chunk {chunk}")
    dev = _device_call(zg, x, window)
    _, rel = errors(out.double().numpy(), dev.double().numpy())
    assert rel <= 1e-3, rel


def test_host_call_pageable_memory(zg):
    """Without page-locked memory the copies do not overlap, but the result is the same."""
    x = _inputs(1, 600, 32, 8, seed=3, pin=False)
    out = zg.swa_prefill_host(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=128,
                              rotary_dim=42, theta=1e4, chunk_tokens=200,
                              out=torch.empty(1, 600, 32, 128, dtype=torch.bfloat16))
    torch.cuda.synchronize()
    dev = _device_call(zg, x, 128)
    _, rel = errors(out.double().numpy(), dev.double().numpy())
    assert rel <= 1e-3, rel


def test_host_call_rejects(zg):
    x = _inputs(1, 64, 8, 2, seed=1)
    with pytest.raises(zg.ZgError, match="ZG_ERR_SHAPE"):
        zg.swa_prefill_host(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=128,
                            rotary_dim=42, theta=1e4, chunk_tokens=0)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(zg.ZgError, match="ZG_ERR_WORKSPACE"):
        zg.swa_prefill_host(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=128,
                            rotary_dim=42, theta=1e4, chunk_tokens=32, workspace=small)
