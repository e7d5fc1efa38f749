"""Multi-GPU host path on CPU: replicas over a world-size-2 gloo group.

The rollout shards by request (independent replicas, no collective on the
data path); the bench's only cross-rank step is the max of the step times.
Each rank here runs the CPU oracle on its own requests, as a replica would
run the library on its GPU.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    from speculative_decoding_draft_lm_gb300 import inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sh = inputs.small_shape(V=300, H=24, E=16, G=16, F=24, dtype="fp32")
    wl = inputs.Workload("replica_test", sh, 2, 0, (1, 2))
    seeds = bench.replica_seeds(wl, rank)
    w = inputs.make_weights(sh, 0)
    r = inputs.make_requests(sh, seeds)
    tokens = oracle.run(w, r)["tokens"]
    my_ms = 1.0 + rank  # a made-up per-rank step time
    ms = bench.max_over_ranks(my_ms, dist, "cpu")
    gathered = [None] * world
    dist.all_gather_object(gathered, {"seeds": seeds, "tokens": tokens.tolist(), "ms": ms})
    if rank == 0:
        out.put(gathered)
    dist.destroy_process_group()


def test_two_replicas_over_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert set(res[0]["seeds"]).isdisjoint(res[1]["seeds"])  # each replica has its own requests
    assert res[0]["ms"] == res[1]["ms"] == 2.0                  # max over ranks
    assert res[0]["tokens"] != res[1]["tokens"]
    import bench
    assert bench.whole_job_rate(2, 2, 2.0) == pytest.approx(15 * 2 * 2 / 2e-3)


def test_single_process_helpers():
    import bench
    from speculative_decoding_draft_lm_gb300 import inputs
    wl = inputs.WORKLOADS["qwen3_8b_b8_k0"]
    assert bench.replica_seeds(wl, 0) == list(wl.request_seeds)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    ab = bench.alg_bytes(inputs.QWEN3_8B, 1, 0)
    # full-vocabulary correction step: fc2 + bias in bf16, one fp32 base row, fp32 activations
    V, F = 151936, 1024
    assert ab["correct"] == V * F * 2 + V * 2 + V * 4 + F * 4
    assert ab["block"] == ab["lmhead"] + ab["steps"]
