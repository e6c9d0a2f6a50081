"""The multi-rank bookkeeping of bench.py on CPU: two gloo ranks.

Decode shards by batch: every rank runs its own batch of the headline
workload on its own GPU (no collective on the data path), and the reported
value is all ranks' bytes over the slowest rank's time.  These tests run the
same helpers the benchmark uses over a real two-process gloo group."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_34_gb300 import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r = {
            "max": bench.reduce_max(dist, float(rank + 1)),
            "sum": bench.reduce_sum(dist, 10.0 * (rank + 1)),
            "seed": bench.rank_seed(W, rank),
            # rank r moved (r + 1) GB in (2 + r) ms
            "job": bench.whole_job_gbs(dist, (rank + 1) * 10 ** 9, 2.0 + rank),
        }
        out[rank] = r
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks():
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    return dict(out)


def test_reductions_are_max_and_sum(two_ranks):
    for r in (0, 1):
        assert two_ranks[r]["max"] == 2.0
        assert two_ranks[r]["sum"] == 30.0


def test_each_rank_draws_its_own_batch(two_ranks):
    assert two_ranks[0]["seed"] != two_ranks[1]["seed"]


def test_whole_job_value_is_all_bytes_over_the_slowest_rank(two_ranks):
    # 1 GB + 2 GB over the slower rank's 3 ms = 1000 GB/s, on both ranks
    for r in (0, 1):
        gbs, ms_max = two_ranks[r]["job"]
        assert ms_max == 3.0
        assert gbs == pytest.approx(1000.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(None, 5.0) == 5.0
    assert bench.whole_job_gbs(None, 2 * 10 ** 9, 4.0) == (pytest.approx(500.0), 4.0)
    assert torch.distributed.is_available()
