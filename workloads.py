"""Seeded synthetic workloads for the ZGCM-1 attention hot path.

This module only DRAWS inputs; it holds none of the attention arithmetic.  It
is the one module shared by the CPU oracle side (tests, the CPU baseline) and
the CUDA side (tests, bench), so both see bit-identical bf16 inputs.

Recipe (the same for every consumer):
  * a CPU ``torch.Generator`` seeded with ``1000 * config + stream`` where the
    stream is q:1, k:2, v:3, gate:4, w_q:5, w_k:6, outlier mask:7, row sample:8,
    output gradient (backward pass):9;
  * values are drawn in float32 and cast to bf16 with round-to-nearest-even;
    the bf16 tensor is the ground truth handed to both sides;
  * activations ~ N(0, 1); QK-norm weights ~ U[0.5, 1.5] in float32;
  * the long-context case scales 1% of the q and k entries (Bernoulli 0.01 per
    element, stream 7) by 20 before the bf16 cast (heavy-tailed outliers);
  * positions are 0 .. L-1 for every sequence (int32).

Sizes follow the ZGCM-1 attention shape: 32 query heads, 8 KV heads, head_dim
128, a 128-token window, rotary_dim = 2 * floor(0.33 * head_dim / 2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

STREAM = {"q": 1, "k": 2, "v": 3, "gate": 4, "wq": 5, "wk": 6, "outlier": 7, "rows": 8, "dout": 9}
_CHUNK = 1 << 24  # elements drawn per generator call (fixed, so chunking never changes values)


def rotary_dim_for(d: int) -> int:
    """Partial-RoPE width for rotary ratio 0.33: 2 * floor(0.33 * d / 2)."""
    return 2 * int(0.33 * d / 2)


@dataclass(frozen=True)
class PrefillCase:
    name: str
    cfg_id: int
    B: int
    L: int
    Hq: int
    Hkv: int
    d: int
    window: int  # 0 = global (full causal)
    rotary_dim: int
    theta: float
    gated: bool
    eps: float = 1e-6
    outliers: bool = False
    sample_rows: int = 0  # 0 = check every row
    full_batches: tuple = ()  # batches checked on every row in addition to the sample

    @property
    def tokens(self) -> int:
        return self.B * self.L


@dataclass(frozen=True)
class DecodeCase:
    name: str
    cfg_id: int
    B: int
    NL: int
    global_layers: tuple
    Hq: int
    Hkv: int
    d: int
    S: int  # global cache capacity (positions)
    W: int  # ring slots of a local layer
    pos: int  # position of the new token (same for every sequence)
    rotary_dim: int
    theta: float
    eps: float = 1e-6
    is_global: tuple = field(default=())

    def layer_flags(self):
        return [1 if l in self.global_layers else 0 for l in range(self.NL)]


TINY_SWA = PrefillCase("tiny_swa_B1_L512_h4x1_d64", 1, 1, 512, 4, 1, 64, 128, 20, 1e4, True)
SWA_4K = PrefillCase("swa_B4_L4096_h32x8_d128", 2, 4, 4096, 32, 8, 128, 128, 42, 1e4, True,
                     sample_rows=int(0.01 * 3 * 4096), full_batches=(0,))
SWA_256K = PrefillCase("swa_B1_L262144_h32x8_d128_outliers", 3, 1, 262144, 32, 8, 128, 128, 42, 1e6, True,
                       outliers=True, sample_rows=4096)
GLOBAL_64K = PrefillCase("global_B1_L65536_h32x8_d128", 4, 1, 65536, 32, 8, 128, 0, 42, 1e6, False, sample_rows=512)
GLOBAL_256K = PrefillCase("global_B1_L262144_h32x8_d128", 4, 1, 262144, 32, 8, 128, 0, 42, 1e6, False,
                          sample_rows=512)
HYBRID_DECODE = DecodeCase("hybrid_decode_B8_p262143_32L", 5, 8, 32, (5, 11, 17, 23, 29), 32, 8, 128,
                           262144, 128, 262143, 42, 1e6)

# global layers of the 32-layer stack, 0-indexed: five blocks of (5 local + 1 global), then 2 local
ZGCM1_GLOBAL_LAYERS = (5, 11, 17, 23, 29)


def _gen(cfg_id: int, stream: str, salt: int = 0) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * cfg_id + STREAM[stream] + 100000 * salt)
    return g


def _randn_bf16(shape, gen: torch.Generator, outlier_gen: torch.Generator | None = None) -> torch.Tensor:
    """N(0,1) drawn in float32 chunk by chunk, optionally with 1% entries x20, cast to bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32)
        if outlier_gen is not None:
            m = torch.rand(e - s, generator=outlier_gen, dtype=torch.float32) < 0.01
            x = torch.where(m, x * 20.0, x)
        flat[s:e] = x.to(torch.bfloat16)
    return out


def norm_weights(d: int, cfg_id: int, stream: str, n: int = 1, salt: int = 0) -> torch.Tensor:
    g = _gen(cfg_id, stream, salt)
    w = 0.5 + torch.rand((n, d), generator=g, dtype=torch.float32)
    return w[0] if n == 1 else w


def prefill_inputs(c: PrefillCase, salt: int = 0) -> dict:
    """CPU tensors: q, k, v, gate (None when ungated) bf16; pos int32; wq, wk float32."""
    og_q = _gen(c.cfg_id, "outlier", salt) if c.outliers else None
    q = _randn_bf16((c.B, c.L, c.Hq, c.d), _gen(c.cfg_id, "q", salt), og_q)
    og_k = _gen(c.cfg_id, "outlier", salt + 7) if c.outliers else None
    k = _randn_bf16((c.B, c.L, c.Hkv, c.d), _gen(c.cfg_id, "k", salt), og_k)
    v = _randn_bf16((c.B, c.L, c.Hkv, c.d), _gen(c.cfg_id, "v", salt))
    gate = _randn_bf16((c.B, c.L, c.Hq, c.d), _gen(c.cfg_id, "gate", salt)) if c.gated else None
    pos = torch.arange(c.L, dtype=torch.int32).repeat(c.B, 1).contiguous()
    return dict(q=q, k=k, v=v, gate=gate, pos=pos,
                wq=norm_weights(c.d, c.cfg_id, "wq", salt=salt), wk=norm_weights(c.d, c.cfg_id, "wk", salt=salt))


def suppressing_gate(shape, cfg_id: int, salt: int = 0, mean: float = -3.0, std: float = 2.0) -> torch.Tensor:
    """Gate logits that mostly suppress: N(mean, std^2) drawn in float32 (stream gate, salt + 50), cast to
    bf16.  With the default N(-3, 2^2) about half of the entries have sigmoid(g) < 0.05."""
    x = _randn_bf16(shape, _gen(cfg_id, "gate", salt + 50)).float()
    return (x * std + mean).to(torch.bfloat16)


def backward_dout(c: PrefillCase, salt: int = 0) -> torch.Tensor:
    """The output gradient a backward pass of case c receives: [B, L, Hq, d] bf16 ~ N(0, 1)."""
    return _randn_bf16((c.B, c.L, c.Hq, c.d), _gen(c.cfg_id, "dout", salt))


def edge_rows(L: int) -> list:
    """Rows that always get checked: the sequence start, both sides of the window edge, the end."""
    cand = [0, 1, 2, 31, 32, 126, 127, 128, 129, 255, 256, L - 2, L - 1]
    return sorted({i for i in cand if 0 <= i < L})


def sample_rows(c: PrefillCase, salt: int = 0) -> list:
    """Flattened (b * L + i) rows to check: all rows of `full_batches`, a seeded sample elsewhere,
    and the edge rows of every batch.  sample_rows == 0 -> every row."""
    if c.sample_rows == 0:
        return list(range(c.B * c.L))
    rows = set()
    for b in c.full_batches:
        rows.update(range(b * c.L, (b + 1) * c.L))
    others = [b for b in range(c.B) if b not in c.full_batches]
    if others:
        g = _gen(c.cfg_id, "rows", salt)
        per = max(1, c.sample_rows // len(others))
        for b in others:
            idx = torch.randint(0, c.L, (per,), generator=g)
            rows.update(int(b * c.L + i) for i in idx)
    for b in range(c.B):
        rows.update(b * c.L + i for i in edge_rows(c.L))
    return sorted(rows)


def decode_token_inputs(c: DecodeCase, salt: int = 0) -> dict:
    """Per-layer new-token tensors: q, gate [NL,B,Hq,d]; k_new, v_new [NL,B,Hkv,d] bf16;
    wq, wk [NL,d] float32; pos [B] int32; is_global [NL] uint8."""
    cid = c.cfg_id
    return dict(
        q=_randn_bf16((c.NL, c.B, c.Hq, c.d), _gen(cid, "q", salt)),
        k_new=_randn_bf16((c.NL, c.B, c.Hkv, c.d), _gen(cid, "k", salt)),
        v_new=_randn_bf16((c.NL, c.B, c.Hkv, c.d), _gen(cid, "v", salt)),
        gate=_randn_bf16((c.NL, c.B, c.Hq, c.d), _gen(cid, "gate", salt)),
        wq=norm_weights(c.d, cid, "wq", n=c.NL, salt=salt),
        wk=norm_weights(c.d, cid, "wk", n=c.NL, salt=salt),
        pos=torch.full((c.B,), c.pos, dtype=torch.int32),
        is_global=torch.tensor(c.layer_flags(), dtype=torch.uint8),
    )


def cache_shapes(c: DecodeCase) -> dict:
    """Shapes of the decode caches: global [NG,B,Hkv,S,d], ring [NS,B,Hkv,W,d]."""
    ng = len(c.global_layers)
    ns = c.NL - ng
    return dict(glob=(ng, c.B, c.Hkv, c.S, c.d), ring=(ns, c.B, c.Hkv, c.W, c.d))


def decode_caches_cpu(c: DecodeCase, salt: int = 0, batches=None) -> dict:
    """CPU bf16 caches ~ N(0,1) (taken as already-normalised keys and raw values).
    `batches`: draw only these sequences (others are not materialised); the draw of
    sequence b never depends on which other sequences are drawn."""
    sh = cache_shapes(c)
    ng, B, Hkv, S, d = sh["glob"]
    ns = sh["ring"][0]
    batches = list(range(B)) if batches is None else list(batches)
    out = {}
    for name, stream, n_l, slots in (("k_glob", "k", ng, S), ("v_glob", "v", ng, S),
                                    ("k_ring", "k", ns, c.W), ("v_ring", "v", ns, c.W)):
        t = torch.empty((n_l, len(batches), Hkv, slots, d), dtype=torch.bfloat16)
        for bi, b in enumerate(batches):
            g = _gen(c.cfg_id, stream, salt=1 + 1000 * (b + 1) + (0 if "glob" in name else 500))
            t[:, bi] = _randn_bf16((n_l, Hkv, slots, d), g)
        out[name] = t
    return out


def decode_caches_device(c: DecodeCase, device, salt: int = 0) -> dict:
    """Device bf16 caches ~ N(0,1) drawn with a seeded CUDA generator (fast path for the
    full-size case; the oracle receives host copies of the slices it checks, taken
    before the decode step runs)."""
    sh = cache_shapes(c)
    out = {}
    for name, stream, shape in (("k_glob", "k", sh["glob"]), ("v_glob", "v", sh["glob"]),
                                ("k_ring", "k", sh["ring"]), ("v_ring", "v", sh["ring"])):
        g = torch.Generator(device=device)
        g.manual_seed(1000 * c.cfg_id + STREAM[stream] + 100000 * salt + (77 if "glob" in name else 99))
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        for s in range(0, flat.numel(), 1 << 28):
            e = min(flat.numel(), s + (1 << 28))
            flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        out[name] = t
    return out


def to_e4m3(t: torch.Tensor, scale: float) -> torch.Tensor:
    """Storage form of an E4M3 cache drawn from a bf16 one: t * scale rounded to float8_e4m3fn
    (torch's round-to-nearest conversion), chunk by chunk on t's device."""
    out = torch.empty(t.shape, dtype=torch.float8_e4m3fn, device=t.device)
    src, dst = t.reshape(-1), out.view(-1)
    for s in range(0, src.numel(), 1 << 28):
        e = min(src.numel(), s + (1 << 28))
        dst[s:e] = (src[s:e].float() * scale).to(torch.float8_e4m3fn)
    return out


def prefill_inputs_device(c: PrefillCase, device, salt: int = 0) -> dict:
    """Same recipe as prefill_inputs, drawn on the device with a seeded CUDA generator (used
    where the values are only timed, e.g. the benchmark; values differ from the CPU draw)."""
    def draw(shape, stream, outlier_stream=None):
        g = torch.Generator(device=device)
        g.manual_seed(1000 * c.cfg_id + STREAM[stream] + 100000 * salt)
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        og = None
        if outlier_stream is not None:
            og = torch.Generator(device=device)
            og.manual_seed(1000 * c.cfg_id + STREAM["outlier"] + 100000 * salt + outlier_stream)
        for s in range(0, flat.numel(), 1 << 28):
            e = min(flat.numel(), s + (1 << 28))
            x = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
            if og is not None:
                m = torch.rand(e - s, generator=og, device=device) < 0.01
                x = torch.where(m, x * 20.0, x)
            flat[s:e] = x.to(torch.bfloat16)
        return t
    q = draw((c.B, c.L, c.Hq, c.d), "q", 0 if c.outliers else None)
    k = draw((c.B, c.L, c.Hkv, c.d), "k", 7 if c.outliers else None)
    v = draw((c.B, c.L, c.Hkv, c.d), "v")
    gate = draw((c.B, c.L, c.Hq, c.d), "gate") if c.gated else None
    pos = torch.arange(c.L, dtype=torch.int32, device=device).repeat(c.B, 1).contiguous()
    return dict(q=q, k=k, v=v, gate=gate, pos=pos,
                wq=norm_weights(c.d, c.cfg_id, "wq", salt=salt).to(device),
                wk=norm_weights(c.d, c.cfg_id, "wk", salt=salt).to(device))
