"""Host logic of the multi-GPU run on CPU (gloo, world size 2).

The path does not shard: `bench.py --gpus N` runs N independent replicas, one process
per GPU, and reports the whole job's rate from the slowest rank's time.  This checks the
pieces of that protocol that need no GPU: the rendezvous, the barrier and the
max-over-ranks reduction of the timing."""
import json
import os
import socket
import sys

import pytest
import torch
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
    r, w, local = bench.dist_info()
    bench.init_dist(w)
    try:
        bench.barrier(w)
        # each rank's "step time"; the job's time is the slowest rank's
        slowest = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
        bench.barrier(w)
    finally:
        torch.distributed.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "slowest": slowest}, f)


def test_two_replicas_max_over_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d == {"rank": r, "world": world, "local": r, "slowest": 1.5 + (world - 1)}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    bench.barrier(1)
    assert not torch.distributed.is_initialized()
