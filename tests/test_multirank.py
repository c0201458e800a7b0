"""The multi-GPU path of the benchmark is replicas only (the GEMM has no
exchange step): each rank runs its own product and the job's time is the
slowest rank's.  Checked here on the CPU with world-size-2 gloo process
groups: the max-over-ranks reduction, the whole-job throughput, and the
reference arm under torchrun (rank 0 alone prints a line; rank 1 exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from dense_fp16_gemm_f16_gb300 import metrics  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, times[rank], "cpu")
        out[rank] = (ms, bench.job_tflops(world, 8192, 8192, 8192, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world, times = 2, [0.61, 0.73]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, value = res[r]
        assert ms == max(times)                          # every rank sees the slowest rank's time
        assert value == pytest.approx(world * metrics.tflops(8192, 8192, 8192, max(times) * 1e-3))


def test_single_rank_passthrough():
    assert bench.max_over_ranks(None, 1.25, "cpu") == 1.25
    assert bench.job_tflops(1, 2, 3, 4, 1.0) == pytest.approx(metrics.tflops(2, 3, 4, 1e-3))


@pytest.mark.slow
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--shape", "256", "256", "256"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    proc = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, proc.stdout                # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
