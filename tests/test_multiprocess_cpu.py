"""The N > 1 bench path on CPU: two gloo ranks (no GPU).

Requests are independent, so ranks shard the job by each prefilling its own
batch; the only exchange is the timing reduction (max over ranks) outside
the data path.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from invariant_paged_prefill_gb300 import workloads as W
    w, r, local = bench.dist_env()
    ms = bench.max_over_ranks(10.0 + r)  # rank r took 10 + r ms
    seed = bench.rank_seed(r)
    b = W.sweep_point(W.HEADS_A, 2, 40, batch=2, seed_data=seed)
    fl = bench.flops_of(W.HEADS_A, b.q_lens, b.kv_lens)
    value = bench.aggregate_value(fl, w, ms)
    gathered = [None] * world
    dist.all_gather_object(gathered, (r, ms, seed, float(b.q.float().sum()), value))
    results[rank] = gathered
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_weak_scaling_helpers():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert set(res) == {0, 1}
    rows = res[0]
    assert rows == res[1]
    # every rank sees the slowest rank's time
    assert all(ms == 11.0 for _, ms, _, _, _ in rows)
    # ranks prefill different data (their own requests)
    assert rows[0][2] != rows[1][2] and rows[0][3] != rows[1][3]
    # whole-job value: both ranks' work over the slowest time
    assert rows[0][4] == rows[1][4]
