"""Split one decode batch across ranks by sequence (host-side layout only).

Decode is independent per (sequence, KV head), so a batch shards by sequence
with no exchange on the data path (the pages' multi-card layouts keep each
request's KV pages with the card that attends over them): rank r of W takes
sequences r, r + W, r + 2W, ...  Each rank keeps only the pool blocks its
sequences use, renumbered 0 .. n_r - 1 in order of their global ids, so its
block table and slot_mapping point into a compact local pool.  Its outputs are
the rows `seqs` of the whole batch's output.

Nothing here launches a kernel or touches the attention arithmetic; it lays
out caller state (block tables, slots, pools, query rows) the way a serving
runtime would before handing each rank its share.
"""
from __future__ import annotations

import copy

import numpy as np
import torch


def shard_by_sequence(x, rank: int, world: int):
    """Rank `rank`'s share of decode batch `x` (a workloads.PagedInputs on
    the host).  Returns (local inputs, seqs): the local batch holds
    sequences `seqs` (global indices, in order) with a compact pool of the
    blocks they use, and rank r's output row i is the batch's output row
    seqs[i]."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if x.kind != "decode":
        raise ValueError("sequence sharding is laid out for decode batches")
    s, bs = x.num_seqs, x.block_size
    seqs = np.arange(rank, s, world, dtype=np.int64)
    ctx = x.context_lens.numpy().astype(np.int64)
    bt = x.block_table.numpy()
    # the blocks each local sequence reads: its first ceil(L / bs) entries
    used = [bt[b, :(ctx[b] + bs - 1) // bs] for b in seqs]
    blocks = np.unique(np.concatenate(used + [np.zeros(0, bt.dtype)]))
    if blocks.size and (blocks.min() < 0 or blocks.max() >= x.num_blocks):
        raise ValueError("a block table entry in use lies outside the pool")
    local_of = {int(g): i for i, g in enumerate(blocks)}

    y = copy.copy(x)
    nb = max(1, int(blocks.size))
    y.num_seqs = int(seqs.size)
    y.num_blocks = nb
    take = torch.from_numpy(blocks.astype(np.int64))
    shape = (nb,) + tuple(x.k_pool.shape[1:])
    y.k_pool = torch.full(shape, float("nan"), dtype=x.k_pool.dtype)
    y.v_pool = y.k_pool.clone()
    if blocks.size:
        y.k_pool[:blocks.size] = x.k_pool[take]
        y.v_pool[:blocks.size] = x.v_pool[take]
    lbt = np.full((seqs.size, bt.shape[1]), -1, dtype=np.int32)
    for i, b in enumerate(seqs):
        n = (ctx[b] + bs - 1) // bs
        lbt[i, :n] = [local_of[int(g)] for g in bt[b, :n]]
    y.block_table = torch.from_numpy(lbt)
    y.context_lens = x.context_lens[torch.from_numpy(seqs)].clone()
    y.q_lens = x.q_lens[torch.from_numpy(seqs)].clone()
    y.new_lens = x.new_lens[torch.from_numpy(seqs)].clone()
    ql = x.q_lens.numpy().astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(ql)])
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs] + [np.zeros(0, np.int64)])
    y.q = x.q[torch.from_numpy(rows)].clone()
    y.cu_seqlens_q = torch.from_numpy(
        np.concatenate([[0], np.cumsum(ql[seqs])]).astype(np.int32))
    # this step's new tokens of the local sequences, slots renumbered
    nl = x.new_lens.numpy().astype(np.int64)
    ncu = np.concatenate([[0], np.cumsum(nl)])
    toks = np.concatenate([np.arange(ncu[b], ncu[b + 1]) for b in seqs] + [np.zeros(0, np.int64)])
    slots = x.slot_mapping.numpy()[toks]
    lslots = np.array([-1 if sl < 0 else local_of[int(sl) // bs] * bs + int(sl) % bs
                       for sl in slots], dtype=np.int64)
    y.slot_mapping = torch.from_numpy(lslots)
    y.k_new = x.k_new[torch.from_numpy(toks)].clone()
    y.v_new = x.v_new[torch.from_numpy(toks)].clone()
    y.max_context_len = int(y.context_lens.max()) if y.num_seqs else 0
    y.max_seqlen_q = int(y.q_lens.max()) if y.num_seqs else 0
    return y, seqs
