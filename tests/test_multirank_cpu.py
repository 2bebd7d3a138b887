"""The N > 1 path on the host, as world_size-2 gloo process groups on CPU.

The op shards by rows with no exchange, so several GPUs run independent
replicas: bench.py's only multi-rank logic is the barrier, the max over
ranks of the timed region and the whole-job sum of work, and that rank 0
alone prints.  These tests run that logic in two CPU processes."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.Dist(rank, world, rank, "gloo")
    try:
        dist.barrier()
        # rank r "took" 1 + r ms for 10 steps of 1 MB and 100 tokens each
        ms, gbs, tok = bench.whole_job(dist, 1_000_000, 100, 10, 1.0 + rank)
        dist.barrier()
    finally:
        dist.close()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "gbs": gbs, "tok": tok}, f)


def test_whole_job_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:  # every rank sees the slowest rank's time and the summed work
        assert r["ms"] == 2.0
        assert r["gbs"] == pytest.approx(1e6 * 10 * world / 2e-3 / 1e9)
        assert r["tok"] == pytest.approx(100 * 10 * world / 2e-3)


def test_single_process_job_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench
    ms, gbs, _ = bench.whole_job(bench.Dist(0, 1, 0, "gloo"), 2_000_000, 1, 5, 4.0)
    assert ms == 4.0 and gbs == pytest.approx(2e6 * 5 / 4e-3 / 1e9)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched the way the driver launches
    N = 2: rank 0 times the oracle and prints one JSON line, rank 1 exits 0
    without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "norm_static_16x1024"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "norm_static_16x1024"
