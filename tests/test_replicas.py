"""Replica runs of bench.py (one independent cache per GPU, no data-path
collective): the whole-job aggregation and the per-rank inputs, run as two
gloo ranks on the CPU."""
import json
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import synth
    from synth.workloads import WORKLOADS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.replica_workload(WORKLOADS["qwen3_30b_a3b_q4_0"], rank)
    router0 = synth.router_weights(w.seed, 0, 8, 64)
    # rank r took (10 + 7r) ms for 256 tokens
    ms, tokens = bench.aggregate(10.0 + 7.0 * rank, 256, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"seed": w.seed, "ms": ms, "tokens": tokens, "router": router0.tolist()}, f)


def test_two_replicas_aggregate_max_time_and_total_tokens(tmp_path):
    import synth
    synth.build()
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(world)]
    for x in r:
        assert x["ms"] == 17.0 and x["tokens"] == 512  # slowest rank's time, all ranks' tokens
    assert r[0]["seed"] != r[1]["seed"]
    assert not np.array_equal(np.array(r[0]["router"]), np.array(r[1]["router"]))


def test_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(12.5, 100) == (12.5, 100)
