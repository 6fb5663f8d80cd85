"""Gradients of the attention prefill (gated SWA or global), for the backward pass.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only tests/, the smoke check
and bench.py's CPU baseline may use it.

The forward is the definition written out in plain fp64 PyTorch CPU operations
(sources: "ZGCM-1-7B 完全解説", gotosocial explainer, section "アーキテクチャ": QK
RMSNorm, partial RoPE with rotary ratio 0.33, sliding window of 128 tokens on the
local layers, full causal attention on the global layers, element-wise sigmoid gate
on the local layers only; "ZGCM-1: A Fully Open and Extremely Efficient Foundation
Model for Math and Agentic Search", jaehun.me review, section "게이트형 SWA의 동작":
the window includes the token itself):

    q_hat = RoPE(q * (mean(q^2) + eps)^-1/2 * wq, pos)        k_hat likewise with wk
    p_ij  = softmax_j over the window (q_hat_i . k_hat_j / sqrt(d))
    out_i = (sum_j p_ij v_j) * sigmoid(g_i)      (global layers: no sigmoid factor)

and the gradients are those of this function, taken by autograd in fp64 — a
library step, as a matmul would be.  The tests pin them with central finite
differences of the same forward on tiny inputs.  The gradients of the RMSNorm
weights are not part of the interface.
"""
from __future__ import annotations

import torch


def _rope(x: torch.Tensor, pos: torch.Tensor, rotary_dim: int, theta: float) -> torch.Tensor:
    """x [..., L, H, d] with pos [..., L]: rotate pairs (j, j + r/2), j < r/2, by pos * theta^(-2j/r)."""
    h = rotary_dim // 2
    if h == 0:
        return x
    j = torch.arange(h, dtype=torch.float64)
    ang = pos.to(torch.float64)[..., None] * theta ** (-2.0 * j / rotary_dim)  # [..., L, h]
    c, s = torch.cos(ang)[..., None, :], torch.sin(ang)[..., None, :]
    a, b = x[..., :h], x[..., h:2 * h]
    return torch.cat([a * c - b * s, b * c + a * s, x[..., 2 * h:]], dim=-1)


def _norm(x: torch.Tensor, w: torch.Tensor, eps: float) -> torch.Tensor:
    return x * torch.rsqrt((x * x).mean(dim=-1, keepdim=True) + eps) * w


def forward(q, k, v, gate, pos, wq, wk, *, window: int, rotary_dim: int, theta: float, eps: float):
    """fp64 forward; q, gate [B,L,Hq,d]; k, v [B,L,Hkv,d]; gate None for a global layer;
    window <= 0 or >= L means full causal attention."""
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    qh = _rope(_norm(q, wq, eps), pos, rotary_dim, theta)
    kh = _rope(_norm(k, wk, eps), pos, rotary_dim, theta)
    rep = Hq // Hkv
    kh = kh.repeat_interleave(rep, dim=2)  # query head h uses KV head h // rep
    vv = v.repeat_interleave(rep, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qh, kh) / d ** 0.5
    i = torch.arange(L)[:, None]
    jj = torch.arange(L)[None, :]
    mask = jj <= i
    if 0 < window < L:
        mask &= (i - jj) < window
    s = s.masked_fill(~mask, float("-inf"))
    p = torch.softmax(s, dim=-1)
    a = torch.einsum("bhij,bjhd->bihd", p, vv)
    return a * torch.sigmoid(gate) if gate is not None else a


def gradients(q, k, v, gate, pos, wq, wk, dout, *, window: int, rotary_dim: int, theta: float, eps: float):
    """dq, dk, dv, dgate (dgate None for a global layer) of sum(forward * dout), all fp64 numpy-ready tensors."""
    f64 = lambda t: None if t is None else torch.as_tensor(t).to(torch.float64).clone().requires_grad_(True)
    q, k, v, g = f64(q), f64(k), f64(v), f64(gate)
    out = forward(q, k, v, g, torch.as_tensor(pos), torch.as_tensor(wq).double(), torch.as_tensor(wk).double(),
                  window=window, rotary_dim=rotary_dim, theta=theta, eps=eps)
    (out * torch.as_tensor(dout).double()).sum().backward()
    return q.grad, k.grad, v.grad, (g.grad if g is not None else None)
