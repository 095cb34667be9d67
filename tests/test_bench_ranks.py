"""The bench's multi-rank path on CPU: world size 2 over gloo.

Each rank runs a replica of the workload; the job time is the slowest rank's and the
throughput counts every rank's FLOPs.  No GPU is involved.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [2.0, 3.0][rank]  # rank 1 is the slow one
        value, tmax = bench.aggregate_throughput(local, 1e12, 10)
        out[rank] = (value, tmax)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank():
    mp_ctx = mp.get_context("spawn")
    mgr = mp_ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        value, tmax = out[rank]
        assert tmax == 3.0
        # 2 ranks x 10 steps x 1e12 FLOP / 3 s = 6.67 TFLOP/s
        assert value == pytest.approx(2 * 10 * 1e12 / 3.0 / 1e12)


def test_single_process_aggregation():
    import bench
    value, tmax = bench.aggregate_throughput(2.0, 1e12, 10)
    assert tmax == 2.0 and value == pytest.approx(5.0)


REQUIRED = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _check_reference_line(line, world):
    import json
    rec = json.loads(line)
    assert REQUIRED <= set(rec), REQUIRED - set(rec)
    assert rec["impl"] == "reference" and rec["n_gpus"] == world
    assert rec["steps"] == 2 and rec["warmup"] == 1 and rec["value"] > 0 and rec["unit"] == "TFLOP/s"
    assert rec["higher_is_better"] is True and rec["vs_baseline"] is None and rec["dtype"] == "f64"
    assert rec["config"]["workload"] == "b1_h2_n256_d64"
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == rec["value"] and cb["sample"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle and prints one JSON line (CPU only)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "b1_h2_n256_d64",
                        "--steps", "2", "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_torchrun_two_ranks():
    """Launched like the multi-GPU bench (torchrun, 2 ranks, gloo): rank 0 alone runs and
    prints; the other rank exits 0 without output."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
                        "--impl", "reference", "--gpus", "2", "--workload", "b1_h2_n256_d64",
                        "--steps", "2", "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    _check_reference_line(lines[0], 2)
