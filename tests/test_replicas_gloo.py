"""The N>1 path of bench.py on CPU: replicas with a barrier and max-over-ranks
timing (no data-path collective), exercised with world_size 2 over gloo.

The operator shards over the batch (independent sequences); this build runs
independent replicas, so the only cross-rank operations are the barrier and
the MAX reduction of the step time, both tested here without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init("gloo")
    assert dist is not None and dist.get_world_size() == world
    bench.barrier(dist)
    # each rank's "step time"; the reported time must be the slowest rank's
    mine = 1.5 + 2.0 * rank
    got = bench.max_over_ranks(mine, dist)
    bench.barrier(dist)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"mine": mine, "max": got}, f)


def test_max_over_ranks_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    assert [r["max"] for r in res] == [3.5, 3.5]
    assert res[0]["mine"] == 1.5


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    try:
        assert bench.dist_init("gloo") is None
        assert bench.max_over_ranks(2.25, None) == 2.25
        bench.barrier(None)
    finally:
        os.environ.clear()
        os.environ.update(env)


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference` launched like the N>1 driver run: rank 0
    alone times the oracle and prints one JSON line; rank 1 exits 0 silently."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--workload", "tiny_lstm", "--steps", "1", "--warmup", "0",
           "--cpu-budget", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "sequences/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("n", [1, 2, 8])
def test_aggregate_value_is_all_ranks_sequences_over_max_time(n):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_sequences_per_s(20, n, 4.0) == pytest.approx(20 * n / 4e-3)
