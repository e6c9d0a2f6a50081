"""One decode batch split by sequence over two gloo ranks (CPU only).

Decode is independent per sequence, so rank r of W can take sequences r,
r + W, ... with only the pool blocks they read (renumbered into a compact
local pool) and no exchange on the data path.  Each rank here lays out its
share with paged_kv_cache_34_gb300.shard, applies the step's write and runs
the oracle's decode on it; the outputs gathered back into the batch's row
order must equal the single-rank oracle's output bit for bit, and the local
block tables and slots must address exactly the rows the global ones do."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _decode_after_write(x):
    import oracle
    kp, vp = oracle._u16(x.k_pool).copy(), oracle._u16(x.v_pool).copy()
    if x.slot_mapping.numel():
        assert oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size) == oracle.OK
    return oracle.decode(x.q, kp, vp, x.block_table, x.context_lens, x.num_kv_heads,
                         x.block_size, x.scale, dtype=oracle.dtype_code(x.dtype)), kp, vp


def _rank_main(rank, world, port, name, out):
    sys.path.insert(0, ROOT)
    from paged_kv_cache_34_gb300 import shard
    from paged_kv_cache_34_gb300 import workloads as W
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = W.make_inputs(name)  # every rank draws the same batch
        y, seqs = shard.shard_by_sequence(x, rank, world)
        got, kp, vp = _decode_after_write(y)
        # gather (seqs, outputs) on every rank
        parts = [None] * world
        dist.all_gather_object(parts, (seqs, got))
        # the local layout addresses the same K rows as the global one
        bs, ok = x.block_size, True
        for i, b in enumerate(seqs):
            for j in range(int(x.context_lens[b])):
                gl = int(x.block_table[b, j // bs]) * bs + j % bs
                lo = int(y.block_table[i, j // bs]) * bs + j % bs
                ok &= torch.equal(x.k_pool.reshape(-1, *x.k_pool.shape[2:])[gl],
                                  y.k_pool.reshape(-1, *y.k_pool.shape[2:])[lo]) or \
                    j == int(x.context_lens[b]) - 1  # the newest row arrives with the write
        out[rank] = {"parts": parts, "layout_ok": bool(ok), "local_blocks": y.num_blocks,
                     "local_slots_ok": bool((y.slot_mapping < y.num_blocks * bs).all())}
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module", params=["llama7b-decode", "continuous-batching"])
def sharded(request):
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, _free_port(), request.param, out), nprocs=2, join=True)
    return request.param, dict(out)


def test_gathered_outputs_equal_the_single_rank_output_bitwise(sharded):
    sys.path.insert(0, ROOT)
    from paged_kv_cache_34_gb300 import workloads as W
    name, out = sharded
    want, _, _ = _decode_after_write(W.make_inputs(name))
    for r in (0, 1):
        got = np.full_like(want, np.nan)
        for seqs, part in out[r]["parts"]:
            got[seqs] = part
        assert np.array_equal(got, want)


def test_local_layout_is_compact_and_addresses_the_same_rows(sharded):
    sys.path.insert(0, ROOT)
    from paged_kv_cache_34_gb300 import workloads as W
    name, out = sharded
    x = W.make_inputs(name)
    bs = x.block_size
    need = int(((x.context_lens + bs - 1) // bs).sum())
    assert out[0]["local_blocks"] + out[1]["local_blocks"] == need  # no block held twice
    for r in (0, 1):
        assert out[r]["layout_ok"] and out[r]["local_slots_ok"]


def test_rank_takes_every_world_th_sequence():
    sys.path.insert(0, ROOT)
    from paged_kv_cache_34_gb300 import shard
    from paged_kv_cache_34_gb300 import workloads as W
    x = W.make_inputs("tiny-decode")
    seen = []
    for r in range(3):
        y, seqs = shard.shard_by_sequence(x, r, 3)
        assert list(seqs) == list(range(r, x.num_seqs, 3))
        assert torch.equal(y.q, x.q[torch.from_numpy(seqs)])
        seen += list(seqs)
    assert sorted(seen) == list(range(x.num_seqs))
    with pytest.raises(ValueError):
        shard.shard_by_sequence(x, 3, 3)
