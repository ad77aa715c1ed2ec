"""Multi-process (world size 2, gloo on CPU) coverage of the N > 1 bench path.

Decode units (sequence, kv_head) are independent, so the multi-GPU bench runs
replicas with no exchange; what the N > 1 path adds is the split of units
over ranks and the max-over-ranks timing.  These run here without a GPU.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from harness import oracle_decode, small_workload
        from synth import make_inputs
        from synth.workloads import shard_units
        w = small_workload("dist", batch=3, q_heads=8, kv_heads=2, len_range=(20, 90))
        inp = make_inputs(w)
        units = [(b, h) for b in range(w.batch) for h in range(w.kv_heads)]
        mine = [units[i] for i in shard_units(len(units), rank, world)]
        res = oracle_decode(inp, set(mine))
        gathered = [None] * world
        dist.all_gather_object(gathered, {k: (v[0].tolist(), v[1].tolist()) for k, v in res.items()})
        slowest = bench.max_over_ranks(1.0 + rank, world)
        if rank == 0:
            q.put((gathered, slowest))
    finally:
        dist.destroy_process_group()


def test_units_split_over_two_gloo_ranks_cover_everything_once():
    from harness import oracle_decode, small_workload
    from synth import make_inputs
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    gathered, slowest = q.get(timeout=60)
    assert slowest == 2.0                                   # max over ranks of (1.0, 2.0)
    merged = {}
    for part in gathered:
        assert not (set(part) & set(merged))                # no unit twice
        merged.update(part)
    w = small_workload("dist", batch=3, q_heads=8, kv_heads=2, len_range=(20, 90))
    full = oracle_decode(make_inputs(w))
    assert set(merged) == set(full)
    for k, (o, l) in full.items():
        np.testing.assert_array_equal(np.array(merged[k][0]), o)
        np.testing.assert_array_equal(np.array(merged[k][1]), l)


@pytest.mark.parametrize("n,world", [(7, 2), (512, 3), (1, 4), (0, 2)])
def test_shard_units_partitions(n, world):
    from synth.workloads import shard_units
    seen = []
    for r in range(world):
        seen.extend(shard_units(n, r, world))
    assert seen == list(range(n))
