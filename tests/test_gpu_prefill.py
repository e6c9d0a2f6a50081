"""pa_prefill_varlen on the GPU against the fp64 oracle, plus the invariants
the pages fix (packed = alone, decode = last prefill row)."""
import numpy as np
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, gpu_decode, gpu_prefill, gpu_write, new_err,
                      oracle_pools_after_write, oracle_prefill, pa, require_gpu, u16)

pytestmark = gpu


def _run(x_host, rows=None, what=""):
    require_gpu()
    kp, vp = oracle_pools_after_write(x_host)
    want = oracle_prefill(x_host, kp, vp, rows=rows)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    out = gpu_prefill(x, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert_close(out, want, x.dtype, rows=rows, what=what)
    return x, out


def sampled_rows(cu, stride=5):
    """Every stride-th packed row plus each sequence's first/last rows and the
    rows around every 128-row tile edge."""
    cu = list(cu)
    rows = set(range(0, cu[-1], stride))
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        for r in (lo, lo + 1, hi - 2, hi - 1):
            if lo <= r < hi:
                rows.add(r)
        for e in range(lo + 127, hi, 128):
            rows.update(r for r in (e - 1, e, e + 1) if lo <= r < hi)
    return np.array(sorted(rows), dtype=np.int64)


def test_packed_prefill_full_size_sampled_rows():
    # The full packed-prefill workload in the benchmark's launch
    # configuration, checked on a sample of rows the oracle computes.
    x = W.make_inputs("packed-prefill")
    _run(x, rows=sampled_rows(x.cu_seqlens_q.tolist()), what="packed-prefill")


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_varlen_grid(bs, hq, hkv, dtype):
    lengths = [1, 5, 127, 128, 129, 300, 64]
    c = cfg(kind="prefill", hq=hq, hkv=hkv, d=128, bs=bs,
            nb=sum(-(-n // bs) for n in lengths) + 3, dtype=dtype, lengths=lengths)
    _run(W.make_inputs(c, seed=200 + bs + hq), what=f"bs{bs} g{hq // hkv} {dtype}")


@pytest.mark.parametrize("bs", [16, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_varlen_grid_head_dim_64(bs, hq, hkv, dtype):
    # head_dim 64: one 128-byte half per tile row, PV with N = 64.
    lengths = [1, 5, 127, 128, 129, 300, 64]
    c = cfg(kind="prefill", hq=hq, hkv=hkv, d=64, bs=bs,
            nb=sum(-(-n // bs) for n in lengths) + 3, dtype=dtype, lengths=lengths)
    _run(W.make_inputs(c, seed=260 + bs + hq), what=f"d64 bs{bs} g{hq // hkv} {dtype}")


def test_chunked_prefill_head_dim_64():
    lengths = [300, 129, 517, 64]
    qlens = [44, 129, 200, 1]
    c = cfg(kind="prefill", hq=8, hkv=4, d=64, bs=32, nb=60, dtype="bf16",
            lengths=lengths)
    x = W.make_inputs(c, seed=61, q_lens=qlens, new_lens=qlens)
    _run(x, what="chunked d64")


@pytest.mark.parametrize("causal", [True, False])
def test_chunked_prefill_queries_shorter_than_context(causal):
    # q < L: the cache already holds a prefix; the step writes the new chunk
    # and its queries attend bottom-right aligned.
    lengths = [300, 129, 517, 64]
    qlens = [44, 129, 200, 1]
    c = cfg(kind="prefill", hq=8, hkv=4, d=128, bs=32, nb=60, dtype="bf16",
            lengths=lengths, causal=causal)
    x = W.make_inputs(c, seed=51, q_lens=qlens, new_lens=qlens)
    _run(x, what=f"chunked causal={causal}")


@pytest.mark.parametrize("d", [128, 64])
def test_packed_equals_each_sequence_alone_bitwise(d):
    require_gpu()
    lengths = [200, 33, 450, 128]
    x = W.make_inputs(cfg(kind="prefill", hq=4, hkv=4, d=d, bs=64, nb=40,
                          lengths=lengths), seed=53).to("cuda")
    gpu_write(x)
    packed = gpu_prefill(x)
    cu = x.cu_seqlens_q.tolist()
    for b in range(len(lengths)):
        y = x.to("cuda")
        y.q = x.q[cu[b]:cu[b + 1]]
        y.cu_seqlens_q = torch.tensor([0, lengths[b]], dtype=torch.int32, device="cuda")
        y.q_lens = x.q_lens[b:b + 1]
        y.context_lens = x.context_lens[b:b + 1]
        y.block_table = x.block_table[b:b + 1]
        alone = gpu_prefill(y)
        torch.cuda.synchronize()
        assert torch.equal(alone.view(torch.int16), packed[cu[b]:cu[b + 1]].view(torch.int16))


def test_decode_matches_last_prefill_row():
    require_gpu()
    lengths = [90, 640, 257]
    x = W.make_inputs(cfg(kind="prefill", hq=8, hkv=2, d=128, bs=16, nb=80,
                          lengths=lengths), seed=57).to("cuda")
    gpu_write(x)
    pre = gpu_prefill(x)
    last = (x.cu_seqlens_q[1:] - 1).long()
    d = x.to("cuda")
    d.q = x.q[last].contiguous()
    dec = gpu_decode(d, partition_size=128)
    torch.cuda.synchronize()
    assert (dec.double() - pre[last].double()).abs().max().item() <= 1e-2


def test_bad_cu_seqlens_flagged_not_faults():
    require_gpu()
    x = W.make_inputs(cfg(kind="prefill", hq=4, hkv=4, d=128, bs=32, nb=30,
                          lengths=[100, 200]), seed=59).to("cuda")
    gpu_write(x)
    x.cu_seqlens_q = torch.tensor([0, 250, 300], dtype=torch.int32, device="cuda")
    err = new_err()
    pa.pa_prefill_varlen(torch.empty_like(x.q), x.q, x.k_pool, x.v_pool, x.block_table,
                         x.cu_seqlens_q, x.context_lens, scale=x.scale, max_seqlen_q=200,
                         max_context_len=200, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_CU_SEQLENS


def test_bad_block_id_flagged_not_faults():
    require_gpu()
    x = W.make_inputs(cfg(kind="prefill", hq=4, hkv=4, d=128, bs=32, nb=30,
                          lengths=[100, 200]), seed=61)
    bt = x.block_table.clone()
    bt[1, 3] = -5
    xd = x.to("cuda")
    gpu_write(xd)
    xd.block_table = bt.cuda()
    err = new_err()
    out = gpu_prefill(xd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BLOCK_ID
    kp, vp = u16(xd.k_pool), u16(xd.v_pool)
    want = oracle_prefill(x, kp, vp, rows=np.arange(100))
    assert_close(out, want, x.dtype, rows=np.arange(100), what="unaffected sequence")


def _prefill_with_hint(x, max_seqlen_q):
    out = torch.empty_like(x.q)
    pa.pa_prefill_varlen(out, x.q, x.k_pool, x.v_pool, x.block_table, x.cu_seqlens_q,
                         x.context_lens, scale=x.scale, max_seqlen_q=max_seqlen_q,
                         max_context_len=x.max_context_len, causal=x.causal)
    return out


def test_chunked_prefill_workload_full_size_every_row():
    # The chunked-prefill workload (16 sequences, contexts of 2K-8K tokens, 1,
    # 4 or 64 new queries each, GQA 4): every output row against the oracle.
    # The four query heads of a KV head share a tile (rows = token x head),
    # so a sequence's 64 queries fill two tiles.
    x = W.make_inputs("chunked-prefill")
    assert x.max_seqlen_q * (x.num_q_heads // x.num_kv_heads) == 256
    _run(x, what="chunked-prefill")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv,qmax", [(8, 8, 128), (8, 2, 32), (16, 2, 16), (8, 2, 128)])
def test_short_queries_grid(d, dtype, causal, hq, hkv, qmax):
    # Short queries against longer contexts, ragged across block and tile
    # edges.  With qmax x (heads packed per KV head) <= 128 every sequence's
    # rows fit one tile (the launch shape whose softmax starts each row's
    # exponentials from its running max); the last case needs two.
    lengths = [1, 128, 129, 300, 517, 1000, 64]
    qlens = [min(q, qmax) for q in (1, 128, 7, 100, 128, 3, 64)]
    c = cfg(kind="prefill", hq=hq, hkv=hkv, d=d, bs=16 if d == 64 else 128,
            nb=sum(-(-n // 16) for n in lengths) + 8, dtype=dtype, lengths=lengths,
            causal=causal)
    x = W.make_inputs(c, seed=71 + d + hq + hkv, q_lens=qlens, new_lens=qlens)
    _run(x, what=f"short q d{d} {dtype} causal={causal} {hq}/{hkv}")


@pytest.mark.parametrize("boost,dtype,hkv", [(20.0, "bf16", 8), (4.0, "f16", 8),
                                             (20.0, "bf16", 2), (4.0, "f16", 2)])
def test_short_queries_equal_long_query_launch_bitwise(boost, dtype, hkv):
    # max_seqlen_q is an upper bound: a hint above 128 / (heads packed per
    # tile) runs the launch shape built for longer queries on the same
    # inputs, and the two give the same bits -- including rows whose running
    # max jumps by more than the rescale threshold in a later key tile (keys
    # 256..299 scaled up), which makes the early-start softmax redo those
    # rows' exponentials (in some rows of a warp and not others).  With the
    # milder boost the scores stay spread enough for the stated fp16 bound
    # against the oracle; with the strong one a few keys carry each row, and
    # the rounding of P to bf16 alone can exceed that bound, so only the two
    # launches are compared.
    require_gpu()
    lengths = [700, 400, 1000]
    pg = 8 // hkv
    qlens = [min(q, 128 // pg) for q in (64, 128, 5)]
    c = cfg(kind="prefill", hq=8, hkv=hkv, d=128, bs=32, nb=80, dtype=dtype, lengths=lengths)
    x = W.make_inputs(c, seed=73, q_lens=qlens, new_lens=qlens)
    kp = x.k_pool.clone()
    for b in range(len(lengths)):
        for j in range(256, 300):
            blk = int(x.block_table[b, j // 32])
            kp[blk, j % 32] = kp[blk, j % 32] * boost
    x.k_pool = kp
    xd = x.to("cuda")
    gpu_write(xd)
    short = _prefill_with_hint(xd, 128 // pg)
    long = _prefill_with_hint(xd, 128 // pg + 1)
    torch.cuda.synchronize()
    assert torch.equal(short.view(torch.int16), long.view(torch.int16))
    if dtype == "f16":
        kpo, vpo = u16(xd.k_pool), u16(xd.v_pool)
        assert_close(short, oracle_prefill(x, kpo, vpo), x.dtype, what="max jumps")


def test_packed_prefill_gqa_full_size_sampled_rows():
    # The packed-prefill workload's lengths and launch shape with 32 query
    # heads over 8 KV heads (GQA 4), on the sampled rows.
    x = W.make_inputs("packed-prefill", num_kv_heads=8)
    _run(x, rows=sampled_rows(x.cu_seqlens_q.tolist()), what="packed-prefill GQA 4")


def test_mid_size_packed_batch_every_row():
    # Eight sequences of about 1000 tokens packed together, every row of
    # every head against the oracle.
    lengths = [1000, 873, 1111, 960, 1024, 777, 1200, 1050]
    c = cfg(kind="prefill", hq=16, hkv=4, d=128, bs=64,
            nb=sum(-(-n // 64) for n in lengths) + 4, dtype="bf16", lengths=lengths)
    _run(W.make_inputs(c, seed=91), what="mid-size packed")


def _expanded_heads(x, g):
    """The same batch with every KV head repeated for each of its g query
    heads (num_kv_heads = num_q_heads): plain multi-head attention."""
    y = x.to("cuda")
    y.k_pool = x.k_pool.repeat_interleave(g, dim=2).contiguous()
    y.v_pool = x.v_pool.repeat_interleave(g, dim=2).contiguous()
    y.num_kv_heads = x.num_q_heads
    return y


@pytest.mark.parametrize("hq,hkv", [(8, 4), (8, 2), (16, 2), (32, 2), (128, 1), (12, 4)])
@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("chunked", [False, True])
def test_gqa_packed_rows_equal_expanded_heads_bitwise(hq, hkv, d, chunked):
    # The query heads of a KV head share a tile's rows (token x head) when
    # the group is a power of two; each row still sees exactly its own
    # token's keys, in the same tiles and order, so the output equals that
    # of the same batch with the KV heads repeated (one head per tile row
    # block) bit for bit.  A group of 3 runs unpacked.  Lengths cross the
    # packed tiles' 128- and 256-row edges.
    require_gpu()
    g = hq // hkv
    lengths = [300, 129, 517, 64, 33] if chunked else [1, 5, 31, 33, 64, 100, 300]
    qlens = [44, 129, 200, 1, 33] if chunked else lengths
    c = cfg(kind="prefill", hq=hq, hkv=hkv, d=d, bs=32,
            nb=sum(-(-n // 32) for n in lengths) + 3, dtype="bf16", lengths=lengths)
    x = W.make_inputs(c, seed=300 + hq + hkv + d + chunked, q_lens=qlens, new_lens=qlens)
    xd = x.to("cuda")
    gpu_write(xd)
    packed = gpu_prefill(xd)
    expanded = gpu_prefill(_expanded_heads(xd, g))
    torch.cuda.synchronize()
    assert torch.equal(packed.view(torch.int16), expanded.view(torch.int16))
    if hq == 16 and d == 128:
        kp, vp = u16(xd.k_pool), u16(xd.v_pool)
        assert_close(packed, oracle_prefill(x, kp, vp), x.dtype, what=f"GQA {g} packed")
