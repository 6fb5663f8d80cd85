"""Attention backward (gated SWA and global): CUDA path through the C ABI against the
fp64 autograd oracle, every element of dq, dk, dv and dgate.

Two paths.  The ZGCM-1 local-layer shape (d = 128, four query heads per KV head,
window 1..128) and the ZGCM-1 global layer (the same heads, every earlier key, no gate)
run on the tensor cores with bf16 MMA operands; every other shape runs in fp32 on the
CUDA cores.

Tolerance of the tensor-core path: the prefill's own bar, rel-L2 <= 1e-2 and max-abs
<= 2e-2 relative to the gradient's largest element.  Its operands q_hat, k_hat, dA,
P and dS are rounded to bf16 (2^-9 relative), which perturbs each score by about
2^-9 |q_hat| |k_hat| / sqrt(128) and each product term by 2^-9; summed over a window
these give relative errors of a few 1e-3.  The exact-zero gradients of window 1 stay
at fp32 rounding because D is formed from the same bf16 dA as dP.

Tolerance of the fp32 path: both sides see the same bf16 inputs; the kernels compute in fp32 and
return fp32 gradients.  The scores |q_hat . k_hat| / sqrt(d) stay below
sqrt(d) * max(wq) * max(wk) (about 25 for weights in [0.5, 1.5]), so an fp32 score
carries an absolute error near 25 * 2^-20 and a softmax weight a relative one of the
same size; 128-term dot products add about 128 * 2^-24.  A relative L2 error of 1e-3
and a max-abs error of 1e-3 * max|reference| leave a wide margin over both while
still failing for any dropped term, wrong sign or transposed operand (those give
relative errors of order one).  Where the exact gradient is zero the relative error is
undefined; there the fp32 residue of a difference of two equal dot products, rounded in
different orders (a few 1e-7), must stay under an absolute floor of 1e-5.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import backward as bw

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3           # fp32 path
MAX_ABS_REL = 1e-3
TC_REL_L2 = 1e-2        # tensor-core path
TC_MAX_ABS_REL = 2e-2
ABS_FLOOR = 1e-5  # where the exact gradient is zero (window 1: ds = p (dA . v - dA . A) with A = v)


@pytest.fixture(scope="module")
def zg():
    import global_attention_fwd_b300 as zg
    return zg


def _tc(c):
    """the shapes the tensor-core path takes: the local layer (window 1..128) and the ungated
    global layer (every earlier key), both with d = 128 and four query heads per KV head"""
    glob = not c.gated and (c.window <= 0 or c.window >= c.L)
    return c.d == 128 and c.Hq == 4 * c.Hkv and (1 <= c.window <= 128 or glob)


def _close(got, ref, what, tc=False):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    ref = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    diff = got - ref
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    ref_norm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / ref_norm) if ref_norm > 0 else 0.0
    mx = float(np.abs(diff).max()) if diff.size else 0.0
    rel_bar, abs_bar = (TC_REL_L2, TC_MAX_ABS_REL) if tc else (REL_L2, MAX_ABS_REL)
    assert mx <= abs_bar * scale + ABS_FLOOR and rel <= rel_bar, \
        f"{what}: max_abs={mx:.3e} (scale {scale:.3e}) rel_l2={rel:.3e}"


def _case(B, L, Hq, Hkv, window, gated, theta=1e4, rotary_dim=42, cfg=50):
    c = workloads.PrefillCase(f"bwd_B{B}_L{L}_{Hq}x{Hkv}_w{window}", cfg, B, L, Hq, Hkv, 128, window, rotary_dim,
                              theta, gated)
    inp = workloads.prefill_inputs(c)
    inp["dout"] = workloads.backward_dout(c)
    return c, inp


def _gpu(zg, c, inp):
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    grads = zg.attention_backward(d["q"], d["k"], d["v"], d["gate"], d["pos"], d["wq"], d["wk"], d["dout"],
                                  window=c.window, rotary_dim=c.rotary_dim, theta=c.theta, eps=c.eps)
    torch.cuda.synchronize()
    assert zg.device_status()[0] == 0
    return grads


def _oracle(c, inp, sl=None):
    """oracle gradients, optionally of the token slice sl of every sequence"""
    x = {k: (v[:, sl] if sl is not None and isinstance(v, torch.Tensor) and v.dim() > 1 else v) for k, v in inp.items()}
    return bw.gradients(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], x["dout"], window=c.window,
                        rotary_dim=c.rotary_dim, theta=c.theta, eps=c.eps)


@pytest.mark.parametrize("B,L,Hq,Hkv,window,gated", [
    (2, 300, 8, 2, 128, True),    # the ZGCM-1 local layer: window 128, GQA 4:1, several windows and a tail
    (1, 257, 8, 2, 0, False),     # global layer: every earlier key, no gate (tensor cores: 3 key blocks)
    (2, 300, 4, 1, 0, False),     # global layer, two sequences, ragged last query tile
    (1, 33, 8, 2, 0, False),      # global layer shorter than one query tile
    (1, 190, 4, 2, 0, False),     # global layer, GQA 2:1 (fp32 path)
    (1, 200, 4, 4, 64, True),     # no head sharing
    (2, 150, 8, 1, 200, True),    # window longer than the sequence, GQA 8:1
    (1, 70, 4, 1, 1, True),       # window 1: every query sees only itself (p = 1, dq = dk = 0)
    (1, 130, 8, 2, 128, False),   # window without gate
    (1, 100, 4, 1, 37, True),     # odd window
    (3, 33, 4, 1, 128, True),     # sequences shorter than the window
])
def test_gradients_match_the_oracle(zg, B, L, Hq, Hkv, window, gated):
    c, inp = _case(B, L, Hq, Hkv, window, gated)
    got = _gpu(zg, c, inp)
    ref = _oracle(c, inp)
    for n, g, r in zip(("dq", "dk", "dv", "dgate"), got, ref):
        if r is None:
            assert g is None
            continue
        _close(g, r, f"{c.name} {n}", tc=_tc(c))


def test_full_size_4k_training_shape_on_window_slices(zg):
    # batch 4 x 4096 tokens, 32 / 8 heads, window 128: the launch the benchmark times.  Inside a
    # slice [t0, t1) of one sequence, dq of rows t >= t0 + 127 and dk, dv of rows
    # t0 + 127 <= t <= t1 - 128 depend only on the slice's own tokens (every window they touch,
    # including the softmax rows of the queries that see a key, lies inside it), so the oracle's
    # gradients of the slice alone are exact references for those rows.  A slice that starts or
    # ends the sequence drops the bound on that side.
    c = workloads.SWA_4K
    inp = workloads.prefill_inputs(c)
    inp["dout"] = workloads.backward_dout(c)
    dq, dk, dv, dg = _gpu(zg, c, inp)
    W = c.window
    for b, t0, t1 in ((0, 0, 384), (1, 1700, 2100), (3, c.L - 384, c.L)):
        one = {k: (v[b:b + 1] if isinstance(v, torch.Tensor) and v.dim() > 1 else v) for k, v in inp.items()}
        rq, rk, rv, rg = _oracle(c, one, slice(t0, t1))
        lo = (t0 + W - 1 if t0 > 0 else t0) - t0
        khi = (t1 - W + 1 if t1 < c.L else t1) - t0
        _close(dq[b, t0 + lo:t1], rq[0, lo:], f"dq b{b} [{t0},{t1})", tc=True)
        _close(dg[b, t0 + lo:t1], rg[0, lo:], f"dgate b{b} [{t0},{t1})", tc=True)
        _close(dk[b, t0 + lo:t0 + khi], rk[0, lo:khi], f"dk b{b} [{t0},{t1})", tc=True)
        _close(dv[b, t0 + lo:t0 + khi], rv[0, lo:khi], f"dv b{b} [{t0},{t1})", tc=True)


def test_global_layer_at_the_4k_training_length(zg):
    # the global layer at the pages' training length (4K): one sequence, one KV group of four
    # query heads (the oracle's autograd over the full 4096 x 4096 score matrices stays within
    # seconds); every element of dq, dk, dv; the global layer has no gate
    c, inp = _case(1, 4096, 4, 1, 0, False, theta=1e6)
    got = _gpu(zg, c, inp)
    ref = _oracle(c, inp)
    assert got[3] is None and ref[3] is None
    for n, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        _close(g, r, f"{c.name} {n}", tc=_tc(c))
