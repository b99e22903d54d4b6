"""The N > 1 path of bench.py on the CPU: world size 2 over gloo.

The decoder forward has no exchange step, so N GPUs run N independent
replicas and the only cross-rank work is the timing barrier, the max of the
ranks' times and rank 0 printing the one result line.  These tests run that
logic as two gloo processes on 127.0.0.1, with no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    reps = bench.Replicas(world, "gloo", None)
    assert reps.dist is not None
    # Each rank reports a different "time"; every rank must see the largest.
    got_max = reps.max(1.5 + rank)
    reps.barrier()
    # The whole-job rate as the bench forms it: all ranks' units over the
    # slowest rank's time.
    units_per_rank = 256
    ms = reps.max(10.0 * (rank + 1))
    value = units_per_rank * world / (ms / 1e3)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got_max, "ms": ms, "value": value}, f)
    reps.close()
    assert reps.dist is None


def test_replicas_gloo_world2(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == 2.5
        assert r["ms"] == 20.0
        assert r["value"] == pytest.approx(256 * 2 / 0.020)
    assert res[0] == res[1]


def test_replicas_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    reps = bench.Replicas(1, "gloo", None)
    assert reps.dist is None
    assert reps.max(3.25) == 3.25
    reps.barrier()
    reps.close()


def test_reference_arm_under_torchrun_world2():
    """torchrun with two ranks: rank 0 alone runs the oracle arm and prints
    one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "toy-decode",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["unit"] == "tokens/s"
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
    # The line names the same workload as our arm's line at N = 2.
    assert rec["config"]["parallelism"] == "replicas x2"
    assert rec["config"]["global_batch"] == 2
    # A reference step is a bounded sample of the workload: here its whole
    # 16 decode tokens; ms_per_step is the measured time of one such step.
    assert rec["tokens_per_step"] == 16
    assert rec["ms_per_step"] == pytest.approx(16 / rec["value"] * 1e3)
