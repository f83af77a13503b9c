"""Data parallelism over the batch (layer_rnn_gb300.dp) on CPU with world size
2 over gloo: every rank runs the step on its shard of the sequences, one
all-reduce sums the weight gradients, and the result equals the whole batch's.

On CPU the ranks' per-shard step is the float64 oracle (the library's kernels
need a GPU); the sharding, the collective and the recombination are the
module's own code, the same that the GPU bench runs with NCCL.
"""

import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from layer_rnn_gb300 import dp  # noqa: E402
from layer_rnn_gb300 import workloads as wl  # noqa: E402


def test_shard_bounds_partition_the_batch():
    for N in (1, 2, 5, 20, 21, 128):
        for world in (1, 2, 3, 4, 7, 8):
            spans = [dp.shard_bounds(N, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0
    with pytest.raises(ValueError):
        dp.shard_bounds(4, 2, 2)


def test_allreduce_is_a_no_op_without_a_process_group():
    import torch
    t = torch.arange(6, dtype=torch.float32)
    assert dp.allreduce_grads(t) is t
    assert torch.equal(t, torch.arange(6, dtype=torch.float32))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CFG = wl.make_config("lstm", 2, True, 4, 5, 3, 4, "f32", 0.3, seed=23)


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    from layer_rnn_gb300 import dp as dpm
    from layer_rnn_gb300 import workloads as wlm
    dist.init_process_group(backend="gloo")
    cfg = CFG
    inp = wlm.make_inputs(cfg)

    def compute(shard):
        out = oracle.run_flat(cfg["mode"], cfg["L"], cfg["bidir"], cfg["I"], cfg["H"],
                              shard["x"], shard["h0"], shard["c0"], shard["w"], shard["dy"],
                              shard["dhy"], shard["dcy"])
        out["dW"] = torch.from_numpy(out["dW"].copy())
        return out

    step = dpm.DataParallelStep(compute, world, rank, dist)
    out = step(inp, cfg["N"])
    # a bf16 buffer: summed in fp32, rounded once
    b = torch.tensor([1.0 + rank, 2 ** -8 * (rank + 1), -3.0], dtype=torch.bfloat16)
    dpm.allreduce_grads(b, dist)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"dW": out["dW"].tolist(), "dx": out["dx"].tolist(),
                   "dh0": out["dh0"].tolist(), "bounds": list(out["bounds"]),
                   "bf16": b.float().tolist()}, f)


def test_two_ranks_sum_to_the_whole_batch(tmp_path):
    import oracle
    import torch.multiprocessing as mp
    world = 2
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    inp = wl.make_inputs(CFG)
    full = oracle.run_flat(CFG["mode"], CFG["L"], CFG["bidir"], CFG["I"], CFG["H"], inp["x"],
                           inp["h0"], inp["c0"], inp["w"], inp["dy"], inp["dhy"], inp["dcy"])
    for r in res:
        # every rank holds the whole batch's weight gradient after the all-reduce
        np.testing.assert_allclose(np.array(r["dW"]), full["dW"], rtol=1e-12, atol=1e-14)
        n0, n1 = r["bounds"]
        np.testing.assert_allclose(np.array(r["dx"]), full["dx"][:, n0:n1], rtol=1e-12,
                                   atol=1e-14)
        np.testing.assert_allclose(np.array(r["dh0"]), full["dh0"][:, n0:n1], rtol=1e-12,
                                   atol=1e-14)
        assert r["bf16"] == [3.0, 3 * 2 ** -8, -6.0]
    assert [r["bounds"] for r in res] == [[0, 3], [3, 5]]
