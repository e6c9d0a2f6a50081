"""Seeded synthetic inputs for the paged-KV attention path.

This module is the only code shared by the CUDA path's callers and the
oracle's tests.  It draws random numbers and lays out the caller-side state
(block tables, the physical pool, the packed query buffer); it holds none of
the attention arithmetic and imports neither the CUDA binding nor the oracle.

Workload shapes follow the five synthetic configurations the library is
measured on (named by what they are):

  tiny-decode          4 seqs, L ~ U[1,128], 8 q / 2 KV heads, D 64, bs 16,
                       64-block pool, permuted block ids, fp16
  llama7b-decode       8 seqs, L ~ U[512,2048], 32/32 heads, D 128, bs 16,
                       8192-block pool, random ids, bf16, new token written
                       through slot_mapping then attended
  continuous-batching  32 seqs, L ~ logU[50,2000], 32/8 heads, D 128, bs 32,
                       shuffled free list over 16384 blocks, fp16
  packed-prefill       16 seqs, q = L ~ U[50,2000], causal, 32/32 heads,
                       D 128, bs 128, 512-block pool, bf16; every token's K/V
                       written through slot_mapping, then attention
  long-context-decode  4 seqs, L ~ U[32768,131072], 64/8 heads, D 128,
                       bs 128, 4096-block pool, bf16, split-KV partitions of
                       512 tokens

and one more shape for the chunked-prefill / multi-token-decode use of the
prefill (q < L, bottom-right causal):

  chunked-prefill      16 seqs, L ~ U[2048,8192], q cycling 1, 4, 64 (the
                       newest q tokens of each context are the queries and
                       this step's writes), causal, 32/8 heads, D 128,
                       bs 128, 1024-block pool, bf16

Values are N(0,1) drawn in fp32 by numpy's PCG64 and rounded to the config
dtype (round-to-nearest-even, by torch's conversion).  Pool rows no sequence
uses hold NaN, so a stray read of an unused slot poisons the output.

Placement (the allocator's job on the pages, outside the hot path): each
sequence takes ceil(capacity / bs) physical blocks popped in order from a
seeded order of the pool, and its logical position p lives in pool row
blocks[p // bs] * bs + p % bs.  Unused block-table entries hold -1.
"""
from __future__ import annotations

import copy
import dataclasses
import math

import numpy as np
import torch

CONFIGS = {
    "tiny-decode": dict(
        kind="decode", num_seqs=4, lengths=("uniform", 1, 128), num_q_heads=8,
        num_kv_heads=2, head_dim=64, block_size=16, num_blocks=64,
        placement="permutation", dtype="f16", write_new_token=False,
        partition_size=0),
    "llama7b-decode": dict(
        kind="decode", num_seqs=8, lengths=("uniform", 512, 2048),
        num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
        num_blocks=8192, placement="sample", dtype="bf16",
        write_new_token=True, partition_size=0),
    "continuous-batching": dict(
        kind="decode", num_seqs=32, lengths=("loguniform", 50, 2000),
        num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
        num_blocks=16384, placement="free_list", dtype="f16",
        write_new_token=False, partition_size=0),
    "packed-prefill": dict(
        kind="prefill", num_seqs=16, lengths=("uniform", 50, 2000),
        num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=128,
        num_blocks=512, placement="permutation", dtype="bf16", causal=True),
    "long-context-decode": dict(
        kind="decode", num_seqs=4, lengths=("uniform", 32768, 131072),
        num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=128,
        num_blocks=4096, placement="permutation", dtype="bf16",
        write_new_token=False, partition_size=512),
    "chunked-prefill": dict(
        kind="prefill", num_seqs=16, lengths=("uniform", 2048, 8192),
        q_lens=("cycle", [1, 4, 64]), num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=128, num_blocks=1024,
        placement="permutation", dtype="bf16", causal=True),
}

# Config order as the workloads are listed; the seed is 1000 + index.
ORDER = ["tiny-decode", "llama7b-decode", "continuous-batching",
         "packed-prefill", "long-context-decode", "chunked-prefill"]

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def default_seed(name: str) -> int:
    return 1000 + ORDER.index(name) if name in ORDER else 4242


def config(name: str, **overrides) -> dict:
    """A copy of a named config with fields overridden (e.g. shorter
    lengths for a quick test of the same shape)."""
    cfg = copy.deepcopy(CONFIGS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


@dataclasses.dataclass
class PagedInputs:
    """Caller-side state for one step of the path (host tensors unless moved
    with ``to``).  Shapes: q [T_q, Hq, D]; k_new/v_new [N_new, Hkv, D];
    k_pool/v_pool [NB, bs, Hkv, D]; block_table [S, max_blocks] int32;
    context_lens, q_lens, new_lens [S] int32; cu_seqlens_q [S+1] int32;
    slot_mapping [N_new] int64."""
    name: str
    seed: int
    kind: str
    dtype: torch.dtype
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float
    causal: bool
    partition_size: int
    context_lens: torch.Tensor
    q_lens: torch.Tensor
    new_lens: torch.Tensor
    cu_seqlens_q: torch.Tensor
    block_table: torch.Tensor
    slot_mapping: torch.Tensor
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    # Host-side upper bounds the caller passes to the library (computed once
    # from the host copies, so reading them never synchronises a device).
    max_context_len: int = 0
    max_seqlen_q: int = 0

    def to(self, device) -> "PagedInputs":
        out = copy.copy(self)
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            if isinstance(v, torch.Tensor):
                setattr(out, f.name, v.to(device))
        return out


def draw_lengths(rng: np.random.Generator, spec, n: int) -> np.ndarray:
    kind, lo, hi = spec
    if kind == "uniform":  # integers in [lo, hi] inclusive
        return rng.integers(lo, hi + 1, size=n).astype(np.int32)
    if kind == "loguniform":  # round(exp(U(ln lo, ln hi))), clamped
        x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    if kind == "fixed":
        return np.full(n, lo, dtype=np.int32)
    if kind == "list":
        return np.asarray(lo, dtype=np.int32)
    raise ValueError(f"unknown length distribution {kind!r}")


def _block_order(rng: np.random.Generator, placement: str, num_blocks: int,
                 needed: int) -> np.ndarray:
    if placement == "identity":
        return np.arange(num_blocks, dtype=np.int64)
    if placement == "permutation":
        return rng.permutation(num_blocks)
    if placement == "sample":  # random sample without replacement
        return rng.choice(num_blocks, size=needed, replace=False)
    if placement == "free_list":  # a shuffled free list, popped from the front
        free = np.arange(num_blocks, dtype=np.int64)
        rng.shuffle(free)
        return free
    raise ValueError(f"unknown placement {placement!r}")


def _normal(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    x = rng.standard_normal(size=int(np.prod(shape)), dtype=np.float32)
    return torch.from_numpy(x).reshape(shape).to(dtype)


def make_inputs(name_or_cfg, seed: int | None = None, *, lengths=None,
                q_lens=None, new_lens=None, device="cpu",
                **overrides) -> PagedInputs:
    """Build one step's inputs for a named config (or a config dict).

    ``lengths`` (context lengths) may be given explicitly; ``q_lens`` and
    ``new_lens`` default to the config kind: decode has one query per
    sequence and writes one new token when ``write_new_token``; prefill has
    q = new = context (the whole sequence is written, then attended)."""
    cfg = config(name_or_cfg, **overrides) if isinstance(name_or_cfg, str) \
        else dict(name_or_cfg, **overrides)
    name = cfg.get("name", "custom")
    if seed is None:
        seed = default_seed(name)
    rng = np.random.Generator(np.random.PCG64(seed))
    s = int(cfg["num_seqs"])
    hq, hkv, d = cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    bs, nb = cfg["block_size"], cfg["num_blocks"]
    dtype = TORCH_DTYPES[cfg["dtype"]]

    ctx = (np.asarray(lengths, dtype=np.int32) if lengths is not None
           else draw_lengths(rng, cfg["lengths"], s))
    assert ctx.shape == (s,)
    if cfg["kind"] == "decode":
        ql = np.ones(s, np.int32) if q_lens is None else np.asarray(q_lens, np.int32)
        if new_lens is None:
            nl = np.minimum(ctx, 1).astype(np.int32) if cfg.get("write_new_token") \
                else np.zeros(s, np.int32)
        else:
            nl = np.asarray(new_lens, np.int32)
    else:
        if q_lens is not None:
            ql = np.asarray(q_lens, np.int32)
        elif cfg.get("q_lens"):  # ("cycle", [a, b, ...]): sequence b gets entry b % len
            vals = cfg["q_lens"][1]
            ql = np.minimum(np.array([vals[b % len(vals)] for b in range(s)], np.int32), ctx)
        else:
            ql = ctx.copy()
        nl = ql.copy() if new_lens is None else np.asarray(new_lens, np.int32)
    assert np.all(nl <= ctx)

    # Placement: block-table capacity from the distribution's maximum length.
    max_len = int(cfg["lengths"][2]) if cfg["lengths"][0] in ("uniform", "loguniform") \
        else int(ctx.max(initial=0))
    max_len = max(max_len, int(ctx.max(initial=0)))
    mbps = max(1, -(-max_len // bs))
    blocks_per_seq = -(-ctx.astype(np.int64) // bs)
    needed = int(blocks_per_seq.sum())
    if needed > nb:
        raise ValueError(f"pool of {nb} blocks cannot hold {needed}")
    order = _block_order(rng, cfg.get("placement", "permutation"), nb, needed)
    block_table = np.full((s, mbps), -1, dtype=np.int32)
    pool_rows = []  # per sequence: pool row of each logical position
    cursor = 0
    for b in range(s):
        nblk = int(blocks_per_seq[b])
        blocks = np.asarray(order[cursor:cursor + nblk], dtype=np.int64)
        cursor += nblk
        block_table[b, :nblk] = blocks
        rows = (np.repeat(blocks * bs, bs) + np.tile(np.arange(bs), nblk))[:ctx[b]]
        pool_rows.append(rows)

    # Values: queries, cached prefix rows, then the rows this step writes.
    total_q = int(ql.sum())
    q = _normal(rng, (total_q, hq, d), dtype)
    k_pool = torch.full((nb, bs, hkv, d), float("nan"), dtype=dtype,
                        device=device)
    v_pool = k_pool.clone()
    prefix_rows = np.concatenate(
        [pool_rows[b][:ctx[b] - nl[b]] for b in range(s)] + [np.zeros(0, np.int64)])
    npre = len(prefix_rows)
    if npre:
        idx = torch.from_numpy(prefix_rows.astype(np.int64)).to(device)
        k_pool.view(nb * bs, hkv, d)[idx] = _normal(rng, (npre, hkv, d), dtype).to(device)
        v_pool.view(nb * bs, hkv, d)[idx] = _normal(rng, (npre, hkv, d), dtype).to(device)
    slots = np.concatenate(
        [pool_rows[b][ctx[b] - nl[b]:ctx[b]] for b in range(s)] + [np.zeros(0, np.int64)])
    nnew = len(slots)
    k_new = _normal(rng, (nnew, hkv, d), dtype)
    v_new = _normal(rng, (nnew, hkv, d), dtype)

    cu = np.zeros(s + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    inputs = PagedInputs(
        name=name, seed=seed, kind=cfg["kind"], dtype=dtype, num_seqs=s,
        num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
        num_blocks=nb, max_blocks_per_seq=mbps, scale=1.0 / math.sqrt(d),
        causal=bool(cfg.get("causal", cfg["kind"] == "prefill")),
        partition_size=int(cfg.get("partition_size", 0)),
        context_lens=torch.from_numpy(ctx.astype(np.int32)),
        q_lens=torch.from_numpy(ql.astype(np.int32)),
        new_lens=torch.from_numpy(nl.astype(np.int32)),
        cu_seqlens_q=torch.from_numpy(cu),
        block_table=torch.from_numpy(block_table),
        slot_mapping=torch.from_numpy(slots.astype(np.int64)),
        q=q, k_new=k_new, v_new=v_new, k_pool=k_pool, v_pool=v_pool,
        max_context_len=int(ctx.max(initial=0)), max_seqlen_q=int(ql.max(initial=0)))
    return inputs.to(device) if str(device) != "cpu" else inputs
