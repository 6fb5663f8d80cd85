"""NumPy full-matrix formulation of the prefill, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Written separately from
``zg_oracle.c`` and structured differently, so the two can check each other:
RoPE is a block-rotation MATRIX applied per position, GQA is an explicit
repeat of the KV heads, the window is an explicit L x L boolean mask, and the
softmax is taken over whole masked rows.

Sources: "ZGCM-1-7B 完全解説" (gotosocial explainer), section "アーキテクチャ";
"ZGCM-1: A Fully Open and Extremely Efficient Foundation Model for Math and
Agentic Search" (jaehun.me review), section "게이트형 SWA의 동작" (a window of
W tokens includes the token itself; the gate multiplies element-wise).
"""
from __future__ import annotations

import numpy as np


def rope_matrix(d: int, r: int, p: float, theta: float) -> np.ndarray:
    """d x d matrix R(p): identity outside [0, r); on [0, r) each pair
    (j, j + r/2) is rotated counter-clockwise by p * theta**(-2j/r)."""
    R = np.eye(d)
    h = r // 2
    for j in range(h):
        a = p * theta ** (-2.0 * j / r)
        R[j, j], R[j, j + h] = np.cos(a), -np.sin(a)
        R[j + h, j], R[j + h, j + h] = np.sin(a), np.cos(a)
    return R


def window_mask(L: int, window: int) -> np.ndarray:
    """M[i, j] True where query i may attend key j."""
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    m = j <= i
    if window > 0:
        m &= (i - j) < window
    return m


def prefill(q, k, v, gate, pos, wq, wk, *, window, rotary_dim, theta, eps):
    """q, gate [B,L,Hq,d]; k, v [B,L,Hkv,d]; pos [B,L]; -> out [B,L,Hq,d] (float64).

    window <= 0: full causal.  gate None: ungated."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    wq = np.asarray(wq, dtype=np.float64)
    wk = np.asarray(wk, dtype=np.float64)

    def norm(x, w):
        return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w

    qn, kn = norm(q, wq), norm(k, wk)
    qr = np.empty_like(qn)
    kr = np.empty_like(kn)
    for b in range(B):
        for i in range(L):
            R = rope_matrix(d, rotary_dim, float(pos[b][i]), theta)
            qr[b, i] = qn[b, i] @ R.T
            kr[b, i] = kn[b, i] @ R.T
    rep = Hq // Hkv
    kr = np.repeat(kr, rep, axis=2)  # [B,L,Hq,d]
    vr = np.repeat(v, rep, axis=2)
    mask = window_mask(L, window)
    out = np.empty((B, L, Hq, d))
    for b in range(B):
        for h in range(Hq):
            S = qr[b, :, h, :] @ kr[b, :, h, :].T / np.sqrt(d)
            S = np.where(mask, S, -np.inf)
            S = S - S.max(axis=1, keepdims=True)
            P = np.exp(S)
            P /= P.sum(axis=1, keepdims=True)
            out[b, :, h, :] = P @ vr[b, :, h, :]
    if gate is not None:
        out = out * (1.0 / (1.0 + np.exp(-np.asarray(gate, dtype=np.float64))))
    return out
