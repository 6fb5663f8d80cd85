"""The algorithmic work counts behind bench.py's roofline fractions, recounted on the CPU
tensor by tensor (what each call must read and write once, what each unmasked pair costs),
so that a wrong count cannot make a kernel look faster or slower than it is."""
import torch

import bench
import workloads

BF16, F32, I32 = 2, 4, 4


def _numel(*shape):
    n = 1
    for s in shape:
        n *= s
    return n


def test_swa_bytes_are_the_tensors_read_and_written_once():
    c = workloads.SWA_256K
    q_gate_out = 3 * _numel(c.B, c.L, c.Hq, c.d) * BF16
    k_v = 2 * _numel(c.B, c.L, c.Hkv, c.d) * BF16
    assert bench.swa_bytes(c) == q_gate_out + k_v


def test_swa_fp8_bytes_count_one_byte_per_qkv_element():
    c = workloads.SWA_256K
    q = _numel(c.B, c.L, c.Hq, c.d)            # E4M3: one byte each
    gate_out = 2 * _numel(c.B, c.L, c.Hq, c.d) * BF16
    k_v = 2 * _numel(c.B, c.L, c.Hkv, c.d)      # E4M3
    assert bench.swa_fp8_bytes(c) == q + gate_out + k_v
    assert bench.swa_fp8_bytes(c) < bench.swa_bytes(c)


def test_traffic_is_reported_only_for_the_sources_it_was_measured_on(tmp_path, monkeypatch):
    """A per-launch DRAM figure from the committed ncu summary counts only while the kernel sources
    hash to the value recorded beside it; any other hash (sources changed since) gives None."""
    import json
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    path.write_text(json.dumps({"kernel_source_hash": bench.kernel_source_hash(),
                                "per_launch_bytes": {"k": 123, "n": None}}))
    assert bench._traffic("k") == 123
    assert bench._traffic("n") is None and bench._traffic("missing") is None
    path.write_text(json.dumps({"kernel_source_hash": "0" * 16, "per_launch_bytes": {"k": 123}}))
    assert bench._traffic("k") is None
    path.unlink()
    assert bench._traffic("k") is None


def test_window_pairs_by_enumeration():
    for L, W in ((1, 128), (100, 128), (300, 128), (4096, 128), (50, 1), (257, 0)):
        c = workloads.PrefillCase("t", 0, 1, L, 4, 1, 128, W, 42, 1e4, True)
        eff = W if 0 < W < L else L
        assert bench.window_pairs(c) == sum(min(i + 1, eff) for i in range(L)), (L, W)


def test_backward_bytes_and_flops():
    for c in (workloads.SWA_4K, workloads.PrefillCase("u", 0, 2, 300, 8, 2, 128, 128, 42, 1e4, False)):
        rows_q, rows_k = _numel(c.B, c.L, c.Hq), _numel(c.B, c.L, c.Hkv)
        inputs = (3 if c.gated else 2) * rows_q * c.d * BF16 + 2 * rows_k * c.d * BF16 + _numel(c.B, c.L) * I32
        outputs = (2 if c.gated else 1) * rows_q * c.d * F32 + 2 * rows_k * c.d * F32
        assert bench.backward_bytes(c) == inputs + outputs, c.name
        # score, dA . v, and the dq, dk, dv updates: five d-long multiply-adds per (query head, key) pair
        pairs = c.B * c.Hq * sum(min(i + 1, c.window) for i in range(c.L))
        assert bench.backward_flops(c) == 5 * 2 * c.d * pairs


def test_global_flops_count_the_causal_triangle():
    c = workloads.PrefillCase("g", 0, 2, 37, 8, 2, 128, 0, 42, 1e4, False)
    mask = torch.tril(torch.ones(c.L, c.L, dtype=torch.bool))
    assert bench.global_flops(c) == 2 * 2 * c.d * c.Hq * c.B * int(mask.sum())


def test_decode_bytes_bf16_and_e4m3():
    c = workloads.HYBRID_DECODE
    ng = len(c.global_layers)
    ns = c.NL - ng
    tok = c.NL * c.B * (3 * c.Hq + 2 * c.Hkv) * c.d * BF16  # q, gate, out and the new k, v rows
    for eb in (2, 1):
        glob = 2 * ng * c.B * c.Hkv * (c.pos + 1) * c.d * eb  # K and V of positions 0..p
        ring = 2 * ns * c.B * c.Hkv * c.W * c.d * eb          # every ring slot
        assert bench.decode_bytes(c, cache_elem_bytes=eb) == glob + ring + tok
    assert bench.decode_bytes(c) == bench.decode_bytes(c, cache_elem_bytes=2)


def test_kv_cache_and_layer_counts():
    c = workloads.GLOBAL_64K
    rows = _numel(c.B, c.L, c.Hkv)
    assert bench.kv_cache_bytes(c) == rows * (2 * c.d * BF16 + 2 * c.d * BF16 + I32)
    s = workloads.SWA_4K
    hidden = s.Hq * s.d
    proj = 2 * s.B * s.L * hidden * (2 * s.Hq + 2 * s.Hkv) * s.d   # q, g (Hq heads) and k, v (Hkv heads)
    oproj = 2 * s.B * s.L * s.Hq * s.d * hidden
    assert bench.layer_gemm_flops(s, hidden) == proj + oproj
