"""The multi-process host path of bench.py on CPU with the gloo backend (world size 2):
the max-over-ranks timing, the whole-job throughput, and the reference arm under
torchrun (rank 0 alone runs and prints; the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # rank r reports (10 + r) ms for the step and (5 - r) ms for its SWA part
        total, swa = bench.max_over_ranks([10.0 + rank, 5.0 - rank], torch.device("cpu"))
        out[rank] = (total, swa, bench.job_tokens_per_s(ws, 1000, 2, swa))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    ws, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(ws, port, out), nprocs=ws, start_method="spawn", join=True)
        res = dict(out)
    for rank in range(ws):
        total, swa, value = res[rank]
        assert total == 11.0 and swa == 5.0  # every rank sees the slowest rank's times
        assert value == 2 * 1000 * 2 / 5e-3  # all ranks' tokens over the slowest time


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu")) == [3.0, 4.0]


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus",
           "2", "--steps", "1", "--warmup", "0", "--ref-rows", "16"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
