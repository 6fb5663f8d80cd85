#!/usr/bin/env python3
"""Benchmark of the ZGCM-1 attention hot path on B300 (one JSON line on stdout).

One step = one pass of the whole hot path over one batch of synthetic input:
  1. gated sliding-window prefill, B=1, L=262144, 32/8 heads, d=128, window 128
     (the headline: tokens/s),
  2. one hybrid decode step, B=8 sequences at position 262143 through the
     32-layer stack (5 global layers with 256K caches, 27 local 128-slot rings),
  3. global (full causal) prefill, B=1, L=65536, 32/8 heads, d=128.
Inputs are drawn once on the device with seeded generators and stay resident in
HBM; every input is larger than the 126 MB L2, so no flush is needed between
steps.  `value` is the gated-SWA prefill throughput (tokens/s summed over all
ranks, from CUDA events around that call); `parts` reports every call with its
own roofline.  `e2e` runs the SWA prefill through the C-ABI call on host
buffers (zg_swa_prefill_host): the inputs in pinned host memory, copied in and the
output copied back inside the call and the timed region, chunk by chunk,
overlapped with the kernel.  Outside the step, `parts` also
times the other workloads one by one: the tiny gated SWA prefill (latency, L2
flushed), the B=4 L=4096 gated SWA prefill (L2 flushed), the global prefill at
L=262144 (bf16, and with E4M3 inputs on the E4M3 tensor-core path), the SWA
prefill of the step with E4M3 inputs, the decode
step over E4M3 caches, the cache writer, the whole gated
layer and the backward pass (local layer, and the global layer at the 4K training
shape).  `cpu_baseline` times the fp64 oracle on a slice of
the 256K workload, on the whole tiny configuration and on one decode step of one
sequence, with the host CPU model and thread count.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same per-GPU work (replicas, no
collective on the data path); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "gated-SWA prefill tokens/s @256K; hybrid decode µs/step; % of roofline"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
CSRC = os.path.join(ROOT, "global_attention_fwd_b300", "csrc")


def _peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the kernels changed since."""
    try:
        with open(TRAFFIC_PATH) as f:
            t = json.load(f)
        if t.get("kernel_source_hash") != kernel_source_hash():
            return None
        return t["per_launch_bytes"].get(kernel)
    except Exception:
        return None


# ------------------------------------------------------------------ workloads
SWA = workloads.SWA_256K
DEC = workloads.HYBRID_DECODE
GLB = workloads.GLOBAL_64K


def swa_bytes(c):  # algorithmic HBM bytes: read q, gate, k, v once, write out once
    return c.B * c.L * (3 * c.Hq * c.d * 2 + 2 * c.Hkv * c.d * 2)


def swa_fp8_bytes(c):  # the same with E4M3 q, k, v (one byte per element); gate and out stay bf16
    return c.B * c.L * (c.Hq * c.d * (1 + 2 + 2) + 2 * c.Hkv * c.d)


def global_flops(c):  # 2 matmuls x 2 flop x d per unmasked (row, key, head)
    return 4.0 * c.d * c.Hq * c.B * (c.L * (c.L + 1) / 2)


def decode_bytes(c, cache_elem_bytes=2):  # caches read once (global 0..p, rings all slots), new-token rows, outputs
    ng = len(c.global_layers)
    ns = c.NL - ng
    eb = cache_elem_bytes
    cache = 2 * ng * c.B * c.Hkv * (c.pos + 1) * c.d * eb + 2 * ns * c.B * c.Hkv * c.W * c.d * eb
    tok = c.NL * c.B * (3 * c.Hq + 2 * c.Hkv) * c.d * 2
    return cache + tok


def window_pairs(c) -> int:
    """(query, key) pairs one head of one sequence attends: sum over i of min(i + 1, W)."""
    W = c.window if 0 < c.window < c.L else c.L
    return W * (W + 1) // 2 + (c.L - W) * W


def backward_flops(c) -> float:
    """Algorithmic backward FLOPs: per (query head, key) pair the score, dA . v, and the dq, dk, dv
    updates, each a d-long multiply-add: 10 d."""
    return 10.0 * c.d * window_pairs(c) * c.B * c.Hq


def backward_bytes(c) -> int:
    """HBM bytes a fused backward must move: q, gate, dout in (bf16) and dq, dgate out (fp32) per query
    row; k, v in (bf16) and dk, dv out (fp32) per key row; positions."""
    per_tok = c.Hq * c.d * (3 * 2 + (2 if c.gated else 1) * 4) + c.Hkv * c.d * (2 * 2 + 2 * 4) + 4
    if not c.gated:
        per_tok -= c.Hq * c.d * 2
    return c.B * c.L * per_tok


def layer_gemm_flops(c, hidden):  # q/k/v/g projections and o_proj of one layer
    return 2.0 * c.B * c.L * hidden * (3 * c.Hq + 2 * c.Hkv) * c.d


def kv_cache_bytes(c):  # per (token, KV head) row: read k, v and the position, write k_hat, v
    return c.B * c.L * c.Hkv * (4 * c.d * 2 + 4)


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"zg_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over every rank of the job (identity for one process)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist = torch.distributed
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tokens_per_s(ws: int, tokens: int, steps: int, ms: float) -> float:
    """Whole-job throughput: each of the ws ranks processes `tokens` per step (weak scaling);
    the time is the slowest rank's."""
    return ws * tokens * steps / (ms * 1e-3)


# ---------------------------------------------------------------- oracle arm
def oracle_sample(rows: int, nthreads=None, seed_salt=0):
    """Time the fp64 oracle on `rows` consecutive gated-SWA rows (all heads) from the middle of
    the 256K workload (a slice with the 127-token history each row needs)."""
    import oracle

    c = SWA
    start = c.L // 2
    lo = start - (c.window - 1)
    sl = workloads.PrefillCase("swa_slice", c.cfg_id, 1, rows + c.window - 1, c.Hq, c.Hkv, c.d, c.window,
                               c.rotary_dim, c.theta, True, outliers=True)
    inp = workloads.prefill_inputs(sl, salt=seed_salt)
    inp["pos"] = inp["pos"] + lo
    rr = list(range(c.window - 1, c.window - 1 + rows))
    n = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"], inp["pos"], inp["wq"], inp["wk"],
                        window=c.window, rotary_dim=c.rotary_dim, theta=c.theta, eps=c.eps, rows=rr, nthreads=n)
    dt = time.perf_counter() - t0
    return rows / dt, n, dt


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_tiny(nthreads=None):
    """The fp64 oracle on the whole tiny gated-SWA configuration (B=1, L=512, 4/1 heads, d=64)."""
    import oracle

    c = workloads.TINY_SWA
    inp = workloads.prefill_inputs(c)
    n = nthreads or oracle.default_threads()
    t0 = time.perf_counter()
    oracle.prefill_rows(inp["q"], inp["k"], inp["v"], inp["gate"], inp["pos"], inp["wq"], inp["wk"], window=c.window,
                        rotary_dim=c.rotary_dim, theta=c.theta, eps=c.eps, rows=list(range(c.B * c.L)), nthreads=n)
    dt = time.perf_counter() - t0
    return c.tokens / dt, dt


# bounded stand-in for the decode workload's per-sequence oracle time: the same 32-layer stack
# at position 32767 (32768-slot global caches); the oracle's work grows linearly with the position
DEC_SAMPLE = workloads.DecodeCase("hybrid_decode_B1_p32767_32L", 5, 1, 32, (5, 11, 17, 23, 29), 32, 8, 128,
                                  32768, 128, 32767, 42, 1e6)


def oracle_decode_seq(nthreads=None):
    """Seconds for the fp64 oracle to run one decode step of one sequence of DEC_SAMPLE, and that time
    extrapolated to position 262143 (global-layer work x 8)."""
    import oracle

    c = DEC_SAMPLE
    tok = workloads.decode_token_inputs(c)
    caches = workloads.decode_caches_cpu(c, batches=[0])
    t0 = time.perf_counter()
    oracle.decode_seq(tok["q"][:, 0], tok["k_new"][:, 0], tok["v_new"][:, 0], tok["gate"][:, 0], tok["wq"], tok["wk"],
                      c.layer_flags(), caches["k_glob"][:, 0], caches["v_glob"][:, 0], caches["k_ring"][:, 0],
                      caches["v_ring"][:, 0], p=c.pos, rotary_dim=c.rotary_dim, theta=c.theta, eps=c.eps,
                      nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, dt * (DEC.pos + 1) / (c.pos + 1)


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(rows)
    rates, dts = [], []
    n = None
    for _ in range(args.steps):
        r, n, dt = oracle_sample(rows)
        rates.append(r)
        dts.append(dt)
    value = statistics.median(rates)
    sample = (f"{rows} consecutive query rows x all 32 heads of the gated-SWA 256K workload per step "
              f"(rows 131072.., fp64 C oracle); tokens/s = rows/s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(dts), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # the GPU arm's config (its value is the gated-SWA prefill's tokens/s, as this arm's is)
        "config": {"workload": f"{SWA.name} + {DEC.name} + {GLB.name}", "global_batch": SWA.B, "seq_len": SWA.L,
                   "parallelism": "single GPU", "l2": "no flush: every input is larger than L2"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import global_attention_fwd_b300 as zg

    peaks, peak_kind = _peaks()
    # ---- inputs, resident in HBM
    sx = workloads.prefill_inputs_device(SWA, dev)
    s_out = torch.empty_like(sx["q"])
    gx = workloads.prefill_inputs_device(GLB, dev)
    g_out = torch.empty_like(gx["q"])
    g_ws = torch.empty(zg.global_prefill_workspace_bytes(GLB.B, GLB.L, GLB.Hkv, GLB.d), dtype=torch.uint8, device=dev)
    tok = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in workloads.decode_token_inputs(DEC).items()}
    caches = workloads.decode_caches_device(DEC, dev)
    d_ws = torch.empty(zg.hybrid_decode_workspace_bytes(len(DEC.global_layers), DEC.B, DEC.Hq, DEC.d, DEC.S),
                       dtype=torch.uint8, device=dev)
    d_out = torch.empty_like(tok["q"])
    flags = DEC.layer_flags()

    def swa():
        zg.swa_prefill(sx["q"], sx["k"], sx["v"], sx["gate"], sx["pos"], sx["wq"], sx["wk"], window=SWA.window,
                       rotary_dim=SWA.rotary_dim, theta=SWA.theta, eps=SWA.eps, out=s_out)

    def dec():
        zg.hybrid_decode(tok["q"], tok["k_new"], tok["v_new"], tok["gate"], tok["pos"], tok["wq"], tok["wk"], flags,
                         caches["k_glob"], caches["v_glob"], caches["k_ring"], caches["v_ring"],
                         rotary_dim=DEC.rotary_dim, theta=DEC.theta, eps=DEC.eps, out=d_out, workspace=d_ws)

    def glob():
        zg.global_prefill(gx["q"], gx["k"], gx["v"], gx["pos"], gx["wq"], gx["wk"], rotary_dim=GLB.rotary_dim,
                          theta=GLB.theta, eps=GLB.eps, out=g_out, workspace=g_ws)

    parts = [("swa_prefill", swa, 1), ("hybrid_decode", dec, 2), ("global_prefill", glob, 2)]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for _, fn, _ in parts:
            fn()
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after warm-up")

    ev = {name: [] for name, _, _ in parts}

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = vis.split(",")[local] if vis else str(local)
    with Clocks(smi_index) as clk:
        barrier()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            for name, fn, _ in parts:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev[name].append((a, b))
        t_end.record(stream)
        barrier()
    clocks = clk.summary()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after the timed region")
    total_ms = t_start.elapsed_time(t_end)
    part_ms = {name: [a.elapsed_time(b) for a, b in ev[name]] for name in ev}
    swa_ms = sum(part_ms["swa_prefill"])
    total_ms, swa_ms = max_over_ranks([total_ms, swa_ms], dev)
    value = job_tokens_per_s(ws, SWA.tokens, args.steps, swa_ms)

    # ---- rooflines per part (average launch durations on this stream)
    def avg(name):
        return statistics.mean(part_ms[name]) * 1e-3

    sw_t, dc_t, gl_t = avg("swa_prefill"), avg("hybrid_decode"), avg("global_prefill")
    hbm = peaks["hbm_gbs"]
    # a read-only stream (the decode step's access pattern) runs above the copy figure: measure what
    # a library reduction reads per second from one 20 GiB cache tensor, to put beside the copy peak
    rd_src = caches["k_glob"].view(-1)
    rd = []
    for i in range(4):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        torch.sum(rd_src, dtype=torch.float32)
        b.record(stream)
        torch.cuda.synchronize()
        if i:
            rd.append(a.elapsed_time(b) * 1e-3)
    read_peak = rd_src.numel() * rd_src.element_size() / min(rd) / 1e9
    rl_swa = {"bound": "hbm", "achieved": swa_bytes(SWA) / sw_t / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": swa_bytes(SWA) / sw_t / 1e9 / hbm, "traffic": _traffic("swa_prefill_kernel"),
              "algorithmic_bytes": swa_bytes(SWA)}
    rl_dec = {"bound": "hbm", "achieved": decode_bytes(DEC) / dc_t / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": decode_bytes(DEC) / dc_t / 1e9 / hbm, "traffic": _traffic("decode_attn_kernel"),
              "algorithmic_bytes": decode_bytes(DEC), "read_peak_live": read_peak,
              "frac_of_read_peak": decode_bytes(DEC) / dc_t / 1e9 / read_peak}
    gf = global_flops(GLB)
    rl_glb = {"bound": "tensor", "achieved": gf / gl_t / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": gf / gl_t / 1e12 / peaks["bf16_tflops"],
              "frac_of_sustained": gf / gl_t / 1e12 / peaks["bf16_tflops_sustained"],
              "traffic": _traffic("global_attn_kernel"), "algorithmic_flops": gf}
    shares = {"swa_prefill": sw_t, "hybrid_decode": dc_t, "global_prefill": gl_t}
    dominant = max(shares, key=shares.get)
    top = {"swa_prefill": rl_swa, "hybrid_decode": rl_dec, "global_prefill": rl_glb}[dominant]
    roofline = dict(top, kernel=dominant, peak_source=f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured"
                    else "fallback")

    # ---- e2e: the SWA prefill through the C-ABI call on host buffers (zg_swa_prefill_host): the
    # inputs in page-locked host memory, copied in and the output copied back inside the call, chunk
    # by chunk, overlapped with the kernel
    e2e = None
    if not args.no_e2e:
        host = {k: v.cpu().pin_memory() for k, v in sx.items()}
        host_out = torch.empty(s_out.shape, dtype=s_out.dtype).pin_memory()
        chunk = 16384
        hws = torch.empty(zg.swa_prefill_host_workspace_bytes(SWA.B, SWA.Hq, SWA.Hkv, SWA.d, SWA.window, chunk),
                          dtype=torch.uint8, device=dev)
        n_chunks = (SWA.L + chunk - 1) // chunk
        halo = (n_chunks - 1) * ((SWA.window - 1 + 127) // 128 * 128)  # extra key / value / position rows copied
        kv_row = SWA.Hkv * SWA.d * 2
        h2d = (sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v", "gate", "pos", "wq", "wk")) +
               SWA.B * halo * (2 * kv_row + 4))
        d2h = host_out.numel() * host_out.element_size()

        def e2e_call():
            zg.swa_prefill_host(host["q"], host["k"], host["v"], host["gate"], host["pos"], host["wq"], host["wk"],
                                window=SWA.window, rotary_dim=SWA.rotary_dim, theta=SWA.theta, eps=SWA.eps,
                                out=host_out, chunk_tokens=chunk, workspace=hws)

        e2e_call()
        e_steps = max(1, min(args.steps, 3))
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_call()
        e1.record(stream)
        barrier()
        e_ms = e0.elapsed_time(e1)
        ev_ = torch.tensor([e_ms], dtype=torch.float64, device=dev)
        if ws > 1:
            torch.distributed.all_reduce(ev_, op=torch.distributed.ReduceOp.MAX)
        st_, det_ = zg.device_status()
        if st_ != 0:
            raise RuntimeError(f"device status {st_} detail {det_:#x} after the host-buffer call")
        e2e = {"value": ws * SWA.tokens * e_steps / (ev_.item() * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
               "call": f"zg_swa_prefill_host, pinned host buffers, chunks of {chunk} tokens"}
        del hws

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        r, n, dt = oracle_sample(args.cpu_rows)
        tiny_r, tiny_dt = oracle_tiny(n)
        dec_s, dec_s_full = oracle_decode_seq(n)
        cpu = {"value": r, "unit": "tokens/s", "cores": n, "cpu_model": cpu_model(), "kind": "oracle",
               "sample": f"{args.cpu_rows} consecutive query rows x 32 heads of the gated-SWA 256K workload "
                         f"(rows 131072.., fp64 C oracle, {dt:.1f} s); tokens/s = rows/s",
               "tiny_config": {"workload": workloads.TINY_SWA.name, "value": tiny_r, "unit": "tokens/s",
                               "s": tiny_dt, "sample": "every row of the configuration"},
               "decode_step_per_sequence": {"workload": DEC_SAMPLE.name, "s": dec_s,
                                            "s_at_p262143_extrapolated": dec_s_full,
                                            "s_for_B8_extrapolated": 8 * dec_s_full,
                                            "sample": "one sequence, all 32 layers, at position 32767; the "
                                                      "oracle's global-layer work grows linearly with the "
                                                      "position, so x8 for p = 262143 (labelled extrapolated)"}}

    if args.step_only:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{SWA.name} + {DEC.name} + {GLB.name}", "global_batch": SWA.B * ws,
                       "seq_len": SWA.L, "parallelism": "replicas" if ws > 1 else "single GPU",
                       "l2": "no flush: every input is larger than L2"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * sum(n for _, _, n in parts), "clocks": clocks,
            "parts": {"swa_prefill": {"workload": SWA.name, "ms": sw_t * 1e3, "roofline": rl_swa},
                      "hybrid_decode": {"workload": DEC.name, "us_per_step": dc_t * 1e6, "roofline": rl_dec},
                      "global_prefill": {"workload": GLB.name, "ms": gl_t * 1e3, "roofline": rl_glb}},
            "note": "--step-only: parts outside the step not run",
        }
        if rank == 0:
            print(json.dumps(line), flush=True)
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    # ---- decode caches from a prefill (outside the step): the global 64K layer's k_hat / v
    kc = torch.empty((GLB.B, GLB.Hkv, GLB.L, GLB.d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)

    def kv_write():
        zg.kv_cache_write(gx["k"], gx["v"], gx["pos"], gx["wk"], kc, vc, ring=False, rotary_dim=GLB.rotary_dim,
                          theta=GLB.theta, eps=GLB.eps)

    for _ in range(2):
        kv_write()
    kv_ev = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kv_write()
        b.record(stream)
        kv_ev.append((a, b))
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after the cache writes")
    kv_t = statistics.median(a.elapsed_time(b) for a, b in kv_ev) * 1e-3
    kv_bytes = kv_cache_bytes(GLB)
    kvc = {"workload": f"global layer caches of {GLB.name} ({GLB.B * GLB.L * GLB.Hkv} rows)", "us": kv_t * 1e6,
           "roofline": {"bound": "hbm", "achieved": kv_bytes / kv_t / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": kv_bytes / kv_t / 1e9 / hbm, "traffic": _traffic("kv_cache_kernel"),
                        "algorithmic_bytes": kv_bytes}}

    # ---- a whole gated SWA layer from hidden states (outside the step): the 4K configuration's
    # shapes with hidden = Hq * d, synthetic weights
    C2 = workloads.SWA_4K
    hid = C2.Hq * C2.d
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 * C2.cfg_id + 9)
    mk = lambda *shape, scale=1.0: (torch.randn(*shape, generator=gen, device=dev) * scale).to(torch.bfloat16)
    lh = mk(C2.B, C2.L, hid)
    lw = [mk(hid, n, scale=hid ** -0.5) for n in (C2.Hq * C2.d, C2.Hkv * C2.d, C2.Hkv * C2.d, C2.Hq * C2.d)]
    lwo = mk(C2.Hq * C2.d, hid, scale=(C2.Hq * C2.d) ** -0.5)
    lpos = torch.arange(C2.L, dtype=torch.int32, device=dev).repeat(C2.B, 1).contiguous()
    lnq = torch.ones(C2.d, dtype=torch.float32, device=dev)
    ly = torch.empty_like(lh)
    lws = torch.empty(zg.gated_swa_layer_workspace_bytes(C2.B, C2.L, C2.Hq, C2.Hkv, C2.d), dtype=torch.uint8,
                      device=dev)

    def layer():
        zg.gated_swa_layer(lh, lw[0], lw[1], lw[2], lw[3], lwo, lpos, lnq, lnq, Hq=C2.Hq, Hkv=C2.Hkv, window=C2.window,
                           rotary_dim=C2.rotary_dim, theta=C2.theta, out=ly, workspace=lws)

    for _ in range(3):
        layer()
    l_ev = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer()
        b.record(stream)
        l_ev.append((a, b))
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after the layer")
    l_t = statistics.median(a.elapsed_time(b) for a, b in l_ev) * 1e-3
    l_fl = layer_gemm_flops(C2, hid)
    lay = {"workload": f"{C2.name} hidden {hid}", "ms": l_t * 1e3, "tokens_per_s": C2.B * C2.L / l_t,
           "roofline": {"bound": "tensor", "achieved": l_fl / l_t / 1e12, "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": l_fl / l_t / 1e12 / peaks["bf16_tflops"], "traffic": None,
                        "algorithmic_flops": l_fl,
                        "note": "projection GEMM flops only; the attention inside is HBM-bound"}}

    # ---- the other configurations of the workload set (outside the step), each on its own
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # twice the 126 MB L2

    def time_part(fn, n, warm=3, flush_l2=False):
        """median seconds of n launches on this stream (L2 overwritten before each when flush_l2)"""
        for _ in range(warm):
            fn()
        evs = []
        for _ in range(n):
            if flush_l2:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        st_, det_ = zg.device_status()
        if st_ != 0:
            raise RuntimeError(f"device status {st_} detail {det_:#x}")
        return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e-3

    # config 1: the tiny gated SWA prefill (latency; L2 flushed before every launch)
    T1 = workloads.TINY_SWA
    tx = workloads.prefill_inputs_device(T1, dev)
    t_out = torch.empty_like(tx["q"])
    t1_t = time_part(lambda: zg.swa_prefill(tx["q"], tx["k"], tx["v"], tx["gate"], tx["pos"], tx["wq"], tx["wk"],
                                            window=T1.window, rotary_dim=T1.rotary_dim, theta=T1.theta, eps=T1.eps,
                                            out=t_out), 50, flush_l2=True)
    tiny = {"workload": T1.name, "us": t1_t * 1e6, "tokens_per_s": T1.tokens / t1_t, "l2": "flushed before each launch",
            "roofline": {"bound": "latency", "achieved": swa_bytes(T1) / t1_t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": swa_bytes(T1) / t1_t / 1e9 / hbm, "algorithmic_bytes": swa_bytes(T1),
                         "note": "0.92 MB in one launch: launch and pipeline latency, not bandwidth"}}
    del tx, t_out

    # config 2: gated SWA prefill B=4, L=4096 (L2 flushed before every launch: 470 MB of traffic)
    C2x = workloads.SWA_4K
    x2 = workloads.prefill_inputs_device(C2x, dev)
    o2 = torch.empty_like(x2["q"])
    s4_t = time_part(lambda: zg.swa_prefill(x2["q"], x2["k"], x2["v"], x2["gate"], x2["pos"], x2["wq"], x2["wk"],
                                            window=C2x.window, rotary_dim=C2x.rotary_dim, theta=C2x.theta,
                                            eps=C2x.eps, out=o2), 20, flush_l2=True)
    swa4k = {"workload": C2x.name, "us": s4_t * 1e6, "tokens_per_s": C2x.tokens / s4_t,
             "l2": "flushed before each launch",
             "roofline": {"bound": "hbm", "achieved": swa_bytes(C2x) / s4_t / 1e9, "peak": hbm, "unit": "GB/s",
                          "frac": swa_bytes(C2x) / s4_t / 1e9 / hbm, "traffic": None,
                          "algorithmic_bytes": swa_bytes(C2x)}}
    del x2, o2

    # config 4b: global prefill at L = 262144
    G4b = workloads.GLOBAL_256K
    gbx = workloads.prefill_inputs_device(G4b, dev)
    gb_out = torch.empty_like(gbx["q"])
    gb_ws = torch.empty(zg.global_prefill_workspace_bytes(G4b.B, G4b.L, G4b.Hkv, G4b.d), dtype=torch.uint8,
                        device=dev)
    g4_t = time_part(lambda: zg.global_prefill(gbx["q"], gbx["k"], gbx["v"], gbx["pos"], gbx["wq"], gbx["wk"],
                                               rotary_dim=G4b.rotary_dim, theta=G4b.theta, eps=G4b.eps, out=gb_out,
                                               workspace=gb_ws), 2, warm=1)
    gf4 = global_flops(G4b)
    glob256 = {"workload": G4b.name, "ms": g4_t * 1e3, "tokens_per_s": G4b.tokens / g4_t,
               "roofline": {"bound": "tensor", "achieved": gf4 / g4_t / 1e12, "peak": peaks["bf16_tflops"],
                            "unit": "TFLOP/s", "frac": gf4 / g4_t / 1e12 / peaks["bf16_tflops"],
                            "frac_of_sustained": gf4 / g4_t / 1e12 / peaks["bf16_tflops_sustained"],
                            "traffic": None, "algorithmic_flops": gf4}}
    # the same workload with E4M3 inputs (e4m3(x * 1)) on the E4M3 tensor-core path
    g8 = {n: workloads.to_e4m3(gbx[n], 1.0).view(torch.uint8) for n in ("q", "k", "v")}
    del gb_ws
    g8_ws = torch.empty(zg.global_prefill_fp8_workspace_bytes(G4b.B, G4b.L, G4b.Hkv, G4b.d), dtype=torch.uint8,
                        device=dev)
    g8_t = time_part(lambda: zg.global_prefill_fp8(g8["q"], g8["k"], g8["v"], gbx["pos"], gbx["wq"], gbx["wk"],
                                                   rotary_dim=G4b.rotary_dim, theta=G4b.theta, eps=G4b.eps,
                                                   out=gb_out, workspace=g8_ws), 2, warm=1)
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # measured bf16 peak x the nominal E4M3 : bf16 ratio (4.5 : 2.25)
    glob256_fp8 = {"workload": f"{G4b.name} with E4M3 q, k, v", "ms": g8_t * 1e3, "tokens_per_s": G4b.tokens / g8_t,
                   "roofline": {"bound": "tensor", "achieved": gf4 / g8_t / 1e12, "peak": fp8_peak,
                                "unit": "TFLOP/s", "frac": gf4 / g8_t / 1e12 / fp8_peak,
                                "peak_basis": "measured bf16 burst x 2 (nominal E4M3 : bf16 ratio)",
                                "traffic": None, "algorithmic_flops": gf4}}
    del gbx, gb_out, g8, g8_ws, flush

    # the gated SWA prefill of the step's workload with E4M3 q, k, v (e4m3(x * 1)); gate and out bf16
    sx = workloads.prefill_inputs_device(SWA, dev)
    s8 = {n: workloads.to_e4m3(sx[n], 1.0).view(torch.uint8) for n in ("q", "k", "v")}
    s8_out = torch.empty_like(sx["q"])
    s8_ws = torch.empty(zg.global_prefill_fp8_workspace_bytes(SWA.B, SWA.L, SWA.Hkv, SWA.d), dtype=torch.uint8,
                        device=dev)
    s8_t = time_part(lambda: zg.swa_prefill_fp8(s8["q"], s8["k"], s8["v"], sx["gate"], sx["pos"], sx["wq"], sx["wk"],
                                                window=SWA.window, rotary_dim=SWA.rotary_dim, theta=SWA.theta,
                                                eps=SWA.eps, out=s8_out, workspace=s8_ws), 10)
    s8_by = swa_fp8_bytes(SWA)
    swa_fp8 = {"workload": f"{SWA.name} with E4M3 q, k, v", "ms": s8_t * 1e3, "tokens_per_s": SWA.tokens / s8_t,
               "roofline": {"bound": "hbm", "achieved": s8_by / s8_t / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": s8_by / s8_t / 1e9 / hbm, "traffic": _traffic("swa_prefill_fp8_call"),
                            "traffic_note": "k_hat and V^T pre-passes plus the attention kernel, one call",
                            "algorithmic_bytes": s8_by}}
    del sx, s8, s8_out, s8_ws

    # ---- the decode step over E4M3 caches (outside the step): the same workload, caches stored
    # as e4m3(k_hat * 1) and e4m3(v * 8)
    f8 = {k: workloads.to_e4m3(v, 1.0 if k.startswith("k") else 8.0) for k, v in caches.items()}

    def dec8():
        zg.hybrid_decode_fp8(tok["q"], tok["k_new"], tok["v_new"], tok["gate"], tok["pos"], tok["wq"], tok["wk"],
                             flags, f8["k_glob"], f8["v_glob"], f8["k_ring"], f8["v_ring"], k_scale=1.0, v_scale=8.0,
                             rotary_dim=DEC.rotary_dim, theta=DEC.theta, eps=DEC.eps, out=d_out, workspace=d_ws)

    for _ in range(3):
        dec8()
    f8_ev = []
    for _ in range(10):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dec8()
        b.record(stream)
        f8_ev.append((a, b))
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after the fp8 decode")
    f8_t = statistics.median(a.elapsed_time(b) for a, b in f8_ev) * 1e-3
    f8_by = decode_bytes(DEC, cache_elem_bytes=1)
    dec_fp8 = {"workload": f"{DEC.name} with E4M3 caches", "us_per_step": f8_t * 1e6,
               "roofline": {"bound": "hbm", "achieved": f8_by / f8_t / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": f8_by / f8_t / 1e9 / hbm, "traffic": _traffic("decode_attn_kernel_fp8"),
                            "algorithmic_bytes": f8_by, "frac_of_read_peak": f8_by / f8_t / 1e9 / read_peak}}
    del f8

    # ---- backward of the gated SWA prefill (outside the step): the 4K training shape
    bx = workloads.prefill_inputs_device(C2, dev)
    bdout = torch.randn(C2.B, C2.L, C2.Hq, C2.d, generator=gen, device=dev).to(torch.bfloat16)
    bws = torch.empty(zg.attention_backward_workspace_bytes(C2.B, C2.L, C2.Hq, C2.Hkv, C2.d), dtype=torch.uint8,
                      device=dev)

    def backward():
        return zg.attention_backward(bx["q"], bx["k"], bx["v"], bx["gate"], bx["pos"], bx["wq"], bx["wk"], bdout,
                                     window=C2.window, rotary_dim=C2.rotary_dim, theta=C2.theta, eps=C2.eps,
                                     workspace=bws)

    for _ in range(3):
        backward()
    b_ev = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        backward()
        b.record(stream)
        b_ev.append((a, b))
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} detail {detail:#x} after the backward pass")
    b_t = statistics.median(a.elapsed_time(b) for a, b in b_ev) * 1e-3
    b_fl = backward_flops(C2)
    b_by = backward_bytes(C2)
    b_tr = [_traffic(k) for k in ("bwd_tc_prep_kernel", "bwd_qpass_kernel", "bwd_kpass_kernel")]
    bwd = {"workload": f"{C2.name} backward (dq, dk, dv, dgate), three kernels per call", "ms": b_t * 1e3,
           "tokens_per_s": C2.tokens / b_t,
           "roofline": {"bound": "hbm", "achieved": b_by / b_t / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": b_by / b_t / 1e9 / hbm,
                        "traffic": sum(b_tr) if all(x is not None for x in b_tr) else None,
                        "algorithmic_bytes": b_by},
           "tensor": {"achieved_tflops": b_fl / b_t / 1e12, "peak": peaks["bf16_tflops"],
                      "frac": b_fl / b_t / 1e12 / peaks["bf16_tflops"], "algorithmic_flops": b_fl}}

    # ---- backward of the global layer (outside the step): the 4K training shape, every earlier key
    GB = workloads.PrefillCase("global_backward_B4_L4096_h32x8_d128", 4, 4, 4096, 32, 8, 128, 0, 42, 1e6, False)
    gbx2 = workloads.prefill_inputs_device(GB, dev)
    gdout = torch.randn(GB.B, GB.L, GB.Hq, GB.d, generator=gen, device=dev).to(torch.bfloat16)
    gbws = torch.empty(zg.attention_backward_workspace_bytes(GB.B, GB.L, GB.Hq, GB.Hkv, GB.d), dtype=torch.uint8,
                       device=dev)
    gb_t = time_part(lambda: zg.attention_backward(gbx2["q"], gbx2["k"], gbx2["v"], None, gbx2["pos"], gbx2["wq"],
                                                   gbx2["wk"], gdout, window=0, rotary_dim=GB.rotary_dim,
                                                   theta=GB.theta, eps=GB.eps, workspace=gbws), 5)
    gb_fl = backward_flops(GB)
    bwd_glob = {"workload": f"{GB.name} backward (dq, dk, dv), three kernels per call", "ms": gb_t * 1e3,
                "tokens_per_s": GB.tokens / gb_t,
                "roofline": {"bound": "tensor", "achieved": gb_fl / gb_t / 1e12, "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": gb_fl / gb_t / 1e12 / peaks["bf16_tflops"], "traffic": None,
                             "algorithmic_flops": gb_fl}}
    del gbx2, gdout, gbws

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{SWA.name} + {DEC.name} + {GLB.name}", "global_batch": SWA.B * ws,
                   "seq_len": SWA.L, "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "no flush: every input is larger than L2"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(n for _, _, n in parts),
        "clocks": clocks,
        "parts": {
            "gated_swa_layer": lay,
            "kv_cache_write": kvc,
            "attention_backward": bwd,
            "attention_backward_global": bwd_glob,
            "hybrid_decode_fp8": dec_fp8,
            "tiny_swa_prefill": tiny,
            "swa_prefill_4k": swa4k,
            "global_prefill_256k": glob256,
            "global_prefill_256k_fp8": glob256_fp8,
            "swa_prefill_fp8": swa_fp8,
            "swa_prefill": {"workload": SWA.name, "ms": sw_t * 1e3, "tokens_per_s": SWA.tokens / sw_t,
                            "roofline": rl_swa},
            "hybrid_decode": {"workload": DEC.name, "us_per_step": dc_t * 1e6, "roofline": rl_dec},
            "global_prefill": {"workload": GLB.name, "ms": gl_t * 1e3, "tokens_per_s": GLB.tokens / gl_t,
                               "roofline": rl_glb},
        },
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_profile_case(args):
    """A small case of one kernel for ncu captures (warm-up launch + `--steps` launches)."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import global_attention_fwd_b300 as zg

    kind = args.profile_case
    if kind == "swa":
        c = workloads.PrefillCase("swa_B1_L65536_profile", 3, 1, 65536, 32, 8, 128, 128, 42, 1e6, True, outliers=True)
        x = workloads.prefill_inputs_device(c, dev)
        out = torch.empty_like(x["q"])

        def fn():
            zg.swa_prefill(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=128,
                           rotary_dim=c.rotary_dim, theta=c.theta, out=out)
    elif kind == "global":
        c = workloads.PrefillCase("global_B1_L16384_profile", 4, 1, 16384, 32, 8, 128, 0, 42, 1e6, False)
        x = workloads.prefill_inputs_device(c, dev)
        out = torch.empty_like(x["q"])
        ws = torch.empty(zg.global_prefill_workspace_bytes(1, c.L, 8, 128), dtype=torch.uint8, device=dev)

        def fn():
            zg.global_prefill(x["q"], x["k"], x["v"], x["pos"], x["wq"], x["wk"], rotary_dim=c.rotary_dim,
                              theta=c.theta, out=out, workspace=ws)
    elif kind == "global8":
        c = workloads.PrefillCase("global_fp8_B1_L16384_profile", 4, 1, 16384, 32, 8, 128, 0, 42, 1e6, False)
        x = workloads.prefill_inputs_device(c, dev)
        x8 = {n: workloads.to_e4m3(x[n], 1.0).view(torch.uint8) for n in ("q", "k", "v")}
        out = torch.empty_like(x["q"])
        ws = torch.empty(zg.global_prefill_fp8_workspace_bytes(1, c.L, 8, 128), dtype=torch.uint8, device=dev)

        def fn():
            zg.global_prefill_fp8(x8["q"], x8["k"], x8["v"], x["pos"], x["wq"], x["wk"], rotary_dim=c.rotary_dim,
                                  theta=c.theta, out=out, workspace=ws)
    elif kind == "swa8":
        c = workloads.PrefillCase("swa_fp8_B1_L65536_profile", 3, 1, 65536, 32, 8, 128, 128, 42, 1e6, True, outliers=True)
        x = workloads.prefill_inputs_device(c, dev)
        x8 = {n: workloads.to_e4m3(x[n], 1.0).view(torch.uint8) for n in ("q", "k", "v")}
        out = torch.empty_like(x["q"])
        ws = torch.empty(zg.global_prefill_fp8_workspace_bytes(1, c.L, 8, 128), dtype=torch.uint8, device=dev)

        def fn():
            zg.swa_prefill_fp8(x8["q"], x8["k"], x8["v"], x["gate"], x["pos"], x["wq"], x["wk"], window=128,
                               rotary_dim=c.rotary_dim, theta=c.theta, out=out, workspace=ws)
    elif kind == "kvcache":
        c = workloads.PrefillCase("kv_cache_B1_L65536_profile", 4, 1, 65536, 32, 8, 128, 0, 42, 1e6, False)
        x = workloads.prefill_inputs_device(c, dev)
        kc = torch.empty((c.B, c.Hkv, c.L, c.d), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)

        def fn():
            zg.kv_cache_write(x["k"], x["v"], x["pos"], x["wk"], kc, vc, ring=False, rotary_dim=c.rotary_dim,
                              theta=c.theta)
    elif kind == "backward":
        c = workloads.PrefillCase("swa_backward_B1_L4096_profile", 2, 1, 4096, 32, 8, 128, 128, 42, 1e4, True)
        x = workloads.prefill_inputs_device(c, dev)
        dout = torch.randn(c.B, c.L, c.Hq, c.d, device=dev).to(torch.bfloat16)
        ws = torch.empty(zg.attention_backward_workspace_bytes(c.B, c.L, c.Hq, c.Hkv, c.d), dtype=torch.uint8,
                         device=dev)

        def fn():
            zg.attention_backward(x["q"], x["k"], x["v"], x["gate"], x["pos"], x["wq"], x["wk"], dout, window=128,
                                  rotary_dim=c.rotary_dim, theta=c.theta, workspace=ws)
    elif kind == "backward_global":
        c = workloads.PrefillCase("global_backward_B1_L4096_profile", 4, 1, 4096, 32, 8, 128, 0, 42, 1e6, False)
        x = workloads.prefill_inputs_device(c, dev)
        dout = torch.randn(c.B, c.L, c.Hq, c.d, device=dev).to(torch.bfloat16)
        ws = torch.empty(zg.attention_backward_workspace_bytes(c.B, c.L, c.Hq, c.Hkv, c.d), dtype=torch.uint8,
                         device=dev)

        def fn():
            zg.attention_backward(x["q"], x["k"], x["v"], None, x["pos"], x["wq"], x["wk"], dout, window=0,
                                  rotary_dim=c.rotary_dim, theta=c.theta, workspace=ws)
    elif kind == "decode8":
        c = workloads.DecodeCase("hybrid_decode_fp8_B1_p131071_profile", 5, 1, 32, (5, 11, 17, 23, 29), 32, 8, 128,
                                 131072, 128, 131071, 42, 1e6)
        tok = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in workloads.decode_token_inputs(c).items()}
        caches = {k: workloads.to_e4m3(v, 1.0 if k[0] == "k" else 8.0)
                  for k, v in workloads.decode_caches_device(c, dev).items()}
        ws = torch.empty(zg.hybrid_decode_workspace_bytes(5, 1, 32, 128, c.S), dtype=torch.uint8, device=dev)
        flags = c.layer_flags()

        def fn():
            zg.hybrid_decode_fp8(tok["q"], tok["k_new"], tok["v_new"], tok["gate"], tok["pos"], tok["wq"], tok["wk"],
                                 flags, caches["k_glob"], caches["v_glob"], caches["k_ring"], caches["v_ring"],
                                 k_scale=1.0, v_scale=8.0, rotary_dim=c.rotary_dim, theta=c.theta, workspace=ws)
    else:
        c = workloads.DecodeCase("hybrid_decode_B1_p131071_profile", 5, 1, 32, (5, 11, 17, 23, 29), 32, 8, 128,
                                 131072, 128, 131071, 42, 1e6)
        tok = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in workloads.decode_token_inputs(c).items()}
        caches = workloads.decode_caches_device(c, dev)
        ws = torch.empty(zg.hybrid_decode_workspace_bytes(5, 1, 32, 128, c.S), dtype=torch.uint8, device=dev)
        flags = c.layer_flags()

        def fn():
            zg.hybrid_decode(tok["q"], tok["k_new"], tok["v_new"], tok["gate"], tok["pos"], tok["wq"], tok["wk"], flags,
                             caches["k_glob"], caches["v_glob"], caches["k_ring"], caches["v_ring"],
                             rotary_dim=c.rotary_dim, theta=c.theta, workspace=ws)
    for _ in range(1 + args.steps):
        fn()
    torch.cuda.synchronize()
    st, detail = zg.device_status()
    print(json.dumps({"profile_case": c.name, "status": st, "detail": detail}))
    return 0 if st == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=16384)
    ap.add_argument("--ref-rows", type=int, default=4096)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step alone: skip the parts measured outside it (for ncu launch lists)")
    ap.add_argument("--profile-case", choices=["swa", "swa8", "global", "global8", "decode", "kvcache", "backward", "backward_global", "decode8"], default=None,
                    help="run only a small case of one kernel (for ncu captures)")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
