"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test states what fixes the expected value: a closed form, an invariant of
the mathematics, a value printed on the pages (tests/golden/), or a second,
structurally different implementation (oracle/brute.py: full L x L mask,
RoPE as a rotation matrix, explicit KV-head repeat).  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads


def _rand_case(rng, B, L, Hq, Hkv, d, gated=True):
    q = rng.standard_normal((B, L, Hq, d))
    k = rng.standard_normal((B, L, Hkv, d))
    v = rng.standard_normal((B, L, Hkv, d))
    gate = rng.standard_normal((B, L, Hq, d)) if gated else None
    pos = np.tile(np.arange(L, dtype=np.int32), (B, 1))
    wq = (0.5 + rng.random(d)).astype(np.float32)
    wk = (0.5 + rng.random(d)).astype(np.float32)
    return q, k, v, gate, pos, wq, wk


def _all_rows(B, L):
    return np.arange(B * L, dtype=np.int64)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("L", [1, 2, 3, 7, 127, 128, 129, 300])
@pytest.mark.parametrize("d,Hq,Hkv", [(8, 2, 2), (64, 4, 1)])
@pytest.mark.parametrize("window", [128, 4, 0])
def test_c_oracle_matches_numpy_brute_force(L, d, Hq, Hkv, window):
    """Two separately written fp64 formulations agree to rounding (1e-11).
    eps = 0.3 so that a dropped or misplaced eps shows."""
    rng = np.random.default_rng(L * 131 + d + window)
    B = 2 if L <= 129 else 1
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    r = workloads.rotary_dim_for(d)
    kw = dict(window=window, rotary_dim=r, theta=1e4, eps=0.3)
    ref = brute.prefill(q, k, v, gate, pos, wq.astype(np.float64), wk.astype(np.float64), **kw)
    got = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, rows=_all_rows(B, L), **kw)
    np.testing.assert_allclose(got.reshape(ref.shape), ref, rtol=0, atol=1e-11)


def test_brute_force_mask_is_the_pages_window():
    """Window W sees W tokens including itself (the window-4 worked example)."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "gate_example.json")) as f:
        g = json.load(f)
    ex = g["window_example"]
    m = brute.window_mask(8, ex["window"])
    assert list(np.nonzero(m[ex["query_index"]])[0]) == ex["keys_seen"]
    assert m.sum(axis=1).tolist() == [1, 2, 3, 4, 4, 4, 4, 4]


# ------------------------------------------------------------- closed forms

def test_window_one_returns_gated_value():
    """W = 1: each query sees only itself, softmax weight 1, so out = v_i * sigmoid(g_i)."""
    rng = np.random.default_rng(1)
    B, L, Hq, Hkv, d = 2, 37, 4, 2, 16
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    got = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, window=1, rotary_dim=4, theta=1e4, eps=1e-6,
                              rows=_all_rows(B, L)).reshape(B, L, Hq, d)
    exp = np.repeat(v, Hq // Hkv, axis=2) / (1.0 + np.exp(-gate))
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-13)


@pytest.mark.parametrize("window", [128, 5, 0])
def test_identical_keys_give_window_mean_of_values(window):
    """Keys that are equal after norm+RoPE (rotated dims zero) give equal scores, so the
    softmax is uniform over J(i): out = mean of v over max(0, i-W+1)..i.  Pins the
    window bounds and the causal edge with a running mean computed here."""
    rng = np.random.default_rng(2)
    B, L, Hq, Hkv, d, r = 1, 300, 4, 1, 64, 20
    q, k, v, _, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d, gated=False)
    base = rng.standard_normal(d)
    base[:r] = 0.0
    k[:] = base
    got = oracle.prefill_rows(q, k, v, None, pos, wq, wk, window=window, rotary_dim=r, theta=1e4, eps=1e-6,
                              rows=_all_rows(B, L)).reshape(B, L, Hq, d)
    csum = np.concatenate([np.zeros((1, d)), np.cumsum(v[0, :, 0, :], axis=0)])
    W = window if window > 0 else L
    for i in range(L):
        lo = max(0, i - W + 1)
        mean = (csum[i + 1] - csum[lo]) / (i + 1 - lo)
        for h in range(Hq):
            np.testing.assert_allclose(got[0, i, h], mean, rtol=0, atol=1e-12)


def test_zero_gate_logits_halve_the_output():
    """sigmoid(0) = 1/2 exactly, so zero gate logits give exactly 0.5 * A."""
    rng = np.random.default_rng(3)
    B, L, Hq, Hkv, d = 1, 200, 4, 1, 64
    q, k, v, _, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d, gated=False)
    kw = dict(window=128, rotary_dim=20, theta=1e4, eps=1e-6, rows=_all_rows(B, L))
    ungated = oracle.prefill_rows(q, k, v, None, pos, wq, wk, **kw)
    gated = oracle.prefill_rows(q, k, v, np.zeros((B, L, Hq, d)), pos, wq, wk, **kw)
    assert np.array_equal(gated, 0.5 * ungated)


def test_printed_gate_example(golden_dir):
    """The pages' worked example: [2.0,-0.5,1.1] (.) sigmoid(g) with sigmoid(g) = [0.9,0.1,0.6]
    gives [1.8,-0.05,0.66].  Built with W = 1 so that A equals the value row exactly."""
    with open(os.path.join(golden_dir, "gate_example.json")) as f:
        g = json.load(f)
    a = np.array(g["attention_output"])
    s = np.array(g["gate_sigmoid"])
    d = a.size
    logits = np.log(s / (1.0 - s))
    q = np.ones((1, 1, 1, d))
    k = np.ones((1, 1, 1, d))
    v = a.reshape(1, 1, 1, d)
    out = oracle.prefill_rows(q, k, v, logits.reshape(1, 1, 1, d), np.zeros((1, 1), np.int32),
                              np.ones(d, np.float32), np.ones(d, np.float32),
                              window=1, rotary_dim=0, theta=1e4, eps=1e-6, rows=[0])
    np.testing.assert_allclose(out.reshape(d), g["gated_output"], rtol=0, atol=1e-12)


def test_window_at_least_length_equals_global_rows():
    """Rows i < W see keys 0..i under both masks: the SWA path (per-row keys) and the
    global path (precomputed keys) of the C oracle must agree there."""
    rng = np.random.default_rng(4)
    B, L, Hq, Hkv, d = 2, 260, 4, 2, 32
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    kw = dict(rotary_dim=10, theta=1e4, eps=1e-6)
    rows = np.array([b * L + i for b in range(B) for i in range(128)], dtype=np.int64)
    swa = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, window=128, rows=rows, **kw)
    glob = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, window=0, rows=rows, **kw)
    np.testing.assert_allclose(swa, glob, rtol=0, atol=1e-13)
    full = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, window=L, rows=_all_rows(B, L), **kw)
    ref = brute.prefill(q, k, v, gate, pos, wq, wk, window=0, **kw)
    np.testing.assert_allclose(full.reshape(ref.shape), ref, rtol=0, atol=1e-11)


# -------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("p", [0, 1, 17, 4095, 262143])
def test_rope_preserves_norm(p):
    rng = np.random.default_rng(p)
    x = rng.standard_normal(128)
    y = oracle.rope(x, 42, p, 1e6)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    assert np.array_equal(y[42:], x[42:])  # dims >= rotary_dim pass through


def test_rope_relative_position_invariance():
    """<R(p+c) q, R(j+c) k> = <R(p) q, R(j) k>: scores depend on p - j only."""
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p, j, c in [(10, 3, 1000), (262143, 262100, -262000), (5, 5, 77)]:
        a = oracle.rope(q, 42, p, 1e6) @ oracle.rope(k, 42, j, 1e6)
        b = oracle.rope(q, 42, p + c, 1e6) @ oracle.rope(k, 42, j + c, 1e6)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_rope_identity_cases_and_first_pair_rotation():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(64)
    assert np.array_equal(oracle.rope(x, 20, 0, 1e4), x)  # position 0: angle 0
    assert np.array_equal(oracle.rope(x, 0, 123, 1e4), x)  # rotary_dim 0: no rotation
    # the first pair has frequency theta^0 = 1 for any theta: e_0 -> (cos p) e_0 + (sin p) e_{r/2}
    e0 = np.zeros(64)
    e0[0] = 1.0
    for theta in (1e4, 1e6):
        y = oracle.rope(e0, 20, 2.5, theta)
        assert abs(y[0] - math.cos(2.5)) < 1e-15 and abs(y[10] - math.sin(2.5)) < 1e-15
        assert np.count_nonzero(y) == 2


def test_attention_is_shift_invariant_in_positions():
    """Adding a constant to every position leaves the output unchanged (RoPE is relative)."""
    rng = np.random.default_rng(7)
    B, L, Hq, Hkv, d = 1, 150, 4, 1, 64
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    kw = dict(window=128, rotary_dim=20, theta=1e4, eps=1e-6, rows=_all_rows(B, L))
    a = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, **kw)
    b = oracle.prefill_rows(q, k, v, gate, pos + 100000, wq, wk, **kw)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)


def test_rotary_dim_zero_is_plain_attention():
    """r = 0: the output equals attention on normalised q, k without any rotation,
    here computed directly with numpy (softmax over the causal window)."""
    rng = np.random.default_rng(8)
    B, L, Hq, Hkv, d, W = 1, 40, 2, 1, 16, 6
    q, k, v, _, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d, gated=False)
    got = oracle.prefill_rows(q, k, v, None, pos, wq, wk, window=W, rotary_dim=0, theta=1e4, eps=0.0,
                              rows=_all_rows(B, L)).reshape(B, L, Hq, d)
    qn = q / np.sqrt((q ** 2).mean(-1, keepdims=True)) * wq
    kn = k / np.sqrt((k ** 2).mean(-1, keepdims=True)) * wk
    for i in range(L):
        js = list(range(max(0, i - W + 1), i + 1))
        for h in range(Hq):
            s = np.array([qn[0, i, h] @ kn[0, j, 0] for j in js]) / math.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            np.testing.assert_allclose(got[0, i, h], p @ v[0, js, 0], rtol=0, atol=1e-12)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(128) * 7.0
    y = oracle.rmsnorm(x, np.ones(128), 0.0)
    assert abs(np.mean(y ** 2) - 1.0) < 1e-14
    np.testing.assert_allclose(oracle.rmsnorm(3.5 * x, np.ones(128), 0.0), y, rtol=0, atol=1e-14)
    w = rng.random(128)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 0.0), y * w, rtol=0, atol=1e-14)


def test_attention_invariant_to_q_k_scale_at_zero_eps():
    rng = np.random.default_rng(10)
    B, L, Hq, Hkv, d = 1, 140, 4, 1, 64
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    kw = dict(window=128, rotary_dim=20, theta=1e4, eps=0.0, rows=_all_rows(B, L))
    a = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, **kw)
    b = oracle.prefill_rows(q * 9.0, k * 0.01, v, gate, pos, wq, wk, **kw)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


# --------------------------------------------------------------------- GQA

def test_gqa_with_replicated_kv_equals_mha():
    rng = np.random.default_rng(11)
    B, L, Hq, Hkv, d = 1, 150, 8, 2, 32
    q, k, v, gate, pos, wq, wk = _rand_case(rng, B, L, Hq, Hkv, d)
    kw = dict(window=128, rotary_dim=10, theta=1e4, eps=1e-6, rows=_all_rows(B, L))
    gqa = oracle.prefill_rows(q, k, v, gate, pos, wq, wk, **kw)
    k_mha = np.repeat(k, Hq // Hkv, axis=2)
    v_mha = np.repeat(v, Hq // Hkv, axis=2)
    mha = oracle.prefill_rows(q, k_mha, v_mha, gate, pos, wq, wk, **kw)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-13)


# ------------------------------------------------------------------ decode

def _khat(k_raw, w, p, r, theta, eps):
    return oracle.rope(oracle.rmsnorm(k_raw, w, eps), r, p, theta)


@pytest.mark.parametrize("p", [299, 50, 0])
def test_decode_step_equals_last_prefill_row(p):
    """A decode step at position p over caches filled with the normalised+rotated keys of
    positions < p reproduces row p of the prefill (SWA layer: window W over the ring,
    slot t mod W; global layer: full cache, slot t).  Stale slots hold garbage that must
    be ignored; the new token's key is returned for the cache write."""
    rng = np.random.default_rng(12 + p)
    L, Hq, Hkv, d, W, r, theta, eps, S = p + 1, 4, 2, 16, 128, 4, 1e4, 1e-6, 320
    is_global = [0, 1, 0]
    NL = 3
    q = rng.standard_normal((NL, L, Hq, d))
    k = rng.standard_normal((NL, L, Hkv, d))
    v = rng.standard_normal((NL, L, Hkv, d))
    gate = rng.standard_normal((NL, L, Hq, d))
    wq = (0.5 + rng.random((NL, d))).astype(np.float32)
    wk = (0.5 + rng.random((NL, d))).astype(np.float32)
    pos = np.arange(L, dtype=np.int32)[None]
    k_glob = rng.standard_normal((1, Hkv, S, d)) * 50  # garbage everywhere first
    v_glob = rng.standard_normal((1, Hkv, S, d)) * 50
    k_ring = rng.standard_normal((2, Hkv, W, d)) * 50
    v_ring = rng.standard_normal((2, Hkv, W, d)) * 50
    gi = si = 0
    expect = np.zeros((NL, Hq, d))
    for l in range(NL):
        glob = is_global[l]
        row = oracle.prefill_rows(q[l][None], k[l][None], v[l][None], None if glob else gate[l][None], pos,
                                  wq[l], wk[l], window=0 if glob else W, rotary_dim=r, theta=theta, eps=eps,
                                  rows=[p])
        expect[l] = row[0]
        for t in range(p):
            for g in range(Hkv):
                kh = _khat(k[l, t, g], wk[l].astype(np.float64), t, r, theta, eps)
                if glob:
                    k_glob[gi, g, t], v_glob[gi, g, t] = kh, v[l, t, g]
                elif t >= p - W + 1:
                    k_ring[si, g, t % W], v_ring[si, g, t % W] = kh, v[l, t, g]
        gi += glob
        si += 1 - glob
    out, khat_new = oracle.decode_seq(q[:, p], k[:, p], v[:, p], gate[:, p], wq, wk, is_global,
                                      k_glob, v_glob, k_ring, v_ring, p=p, rotary_dim=r, theta=theta, eps=eps)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)
    for l in range(NL):
        for g in range(Hkv):
            np.testing.assert_allclose(khat_new[l, g], _khat(k[l, p, g], wk[l].astype(np.float64), p, r, theta, eps),
                                       rtol=0, atol=1e-14)


# ---------------------------------------------------------- printed numbers

def test_kv_cache_footprint_matches_printed_closed_forms(golden_dir):
    with open(os.path.join(golden_dir, "kv_footprint.json")) as f:
        g = json.load(f)
    c = workloads.HYBRID_DECODE
    sh = workloads.cache_shapes(c)
    ng, B, Hkv, S, d = sh["glob"]
    per_tok = 2 * ng * Hkv * d * 2  # K and V, bf16, per sequence
    assert (Hkv, d) == (g["kv_heads"], g["head_dim"])
    assert per_tok == g["hybrid"]["bytes_per_token"]
    assert 2 * c.NL * Hkv * d * 2 == g["full_attention"]["bytes_per_token"]
    assert per_tok * S / 2 ** 30 == g["hybrid"]["gib_at_262144_tokens"]
    assert 2 * c.NL * Hkv * d * 2 * S / 2 ** 30 == g["full_attention"]["gib_at_262144_tokens"]
    assert g["full_attention"]["bytes_per_token"] / per_tok == g["reduction"]


def test_layer_pattern_matches_pages(golden_dir):
    with open(os.path.join(golden_dir, "layer_pattern.json")) as f:
        g = json.load(f)
    assert list(workloads.ZGCM1_GLOBAL_LAYERS) == g["global_layers_0_indexed"]
    assert [x - 1 for x in g["global_layers_1_indexed"]] == g["global_layers_0_indexed"]
    flags = workloads.HYBRID_DECODE.layer_flags()
    assert len(flags) == g["n_layers"] and sum(flags) == 5
    assert [i for i, f in enumerate(flags) if f] == g["global_layers_0_indexed"]


def test_rotary_dim_reading():
    assert workloads.rotary_dim_for(128) == 42
    assert workloads.rotary_dim_for(64) == 20


def test_bf16_inputs_are_read_exactly():
    """bf16 bit patterns reach the oracle unchanged: W = 1 and zero gate logits return 0.5 * v."""
    v = torch.randn(1, 5, 1, 8).to(torch.bfloat16)
    q = torch.randn(1, 5, 1, 8).to(torch.bfloat16)
    gate = torch.zeros(1, 5, 1, 8, dtype=torch.bfloat16)
    out = oracle.prefill_rows(q, q, v, gate, torch.arange(5, dtype=torch.int32)[None], torch.ones(8), torch.ones(8),
                              window=1, rotary_dim=2, theta=1e4, eps=1e-6, rows=list(range(5)))
    np.testing.assert_array_equal(out.reshape(5, 8), 0.5 * v.double().reshape(5, 8).numpy())
