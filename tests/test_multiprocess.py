"""The multi-rank path of bench.py on CPU with the gloo backend, world size 2:
the layer has no exchange between tokens, so N ranks run N replicas and the
only cross-rank step is the reduction of the timing (the slowest rank's time)
into one whole-job rate, printed by rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench as b

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        slowest = b.reduce_max(10.0 + 5.0 * rank)  # rank 1 is the slow one
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest,
                       "value": b.job_throughput(4096, world, slowest)}, f)
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got["slowest"] == 15.0
        assert got["value"] == pytest.approx(2 * 4096 / 0.015)


def test_single_process_needs_no_group():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_throughput(100, 1, 10.0) == pytest.approx(10000.0)


def test_dist_env_reads_torchrun_variables(monkeypatch):
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "8")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (3, 8, 1)


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks launched the way the driver launches N > 1: rank 0 alone runs
    the CPU oracle arm and prints one line; the other rank exits 0."""
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--gpus", "2", "--steps", "3",
                        "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["parallelism"] == "replicas x2"
