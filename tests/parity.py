"""Shared comparison helpers for the GPU parity tests (no attention arithmetic here).

Tolerance (bf16 inputs and outputs, fp32 accumulation): max-abs error <= 2e-2 and
relative L2 error <= 1e-2 over the checked rows, against the fp64 oracle.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 1e-2


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, ref, what=""):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def rows_of(out: torch.Tensor, rows):
    """out [B,L,H,d] (any device) -> float64 numpy [len(rows), H, d] for flattened rows b*L+i."""
    B, L, H, d = out.shape
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=out.device)
    return out.reshape(B * L, H, d).index_select(0, idx).double().cpu().numpy()
