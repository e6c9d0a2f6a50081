"""Pins for the oracle's attention: it must agree with PyTorch's own fp64
scaled_dot_product_attention where paging is the identity, and satisfy the
invariants and special cases the pages and the mathematics fix.  CPU only."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_34_gb300 import workloads as W


def small_cfg(kind="decode", hq=8, hkv=2, d=64, bs=16, nb=64, dtype="f16",
              lengths=("uniform", 1, 100), placement="permutation", seqs=4):
    return dict(kind=kind, num_seqs=seqs, lengths=lengths, num_q_heads=hq,
                num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                placement=placement, dtype=dtype, name="small")


def contiguous_kv(x, b):
    """K, V of sequence b as [Hkv, L, D] fp64, valid only for identity
    placement (a sequence's blocks are consecutive in the pool)."""
    L = int(x.context_lens[b])
    start = int(x.block_table[b, 0]) * x.block_size
    flat_k = x.k_pool.reshape(-1, x.num_kv_heads, x.head_dim)
    flat_v = x.v_pool.reshape(-1, x.num_kv_heads, x.head_dim)
    k = flat_k[start:start + L].double().permute(1, 0, 2)
    v = flat_v[start:start + L].double().permute(1, 0, 2)
    return k, v


def sdpa(q, k, v, scale, causal=False):
    """q [Hq, n, D], k/v [Hkv, L, D] fp64 -> [Hq, n, D] via torch's SDPA
    (grouped heads: query head h reads KV head h // (Hq/Hkv))."""
    out = F.scaled_dot_product_attention(q[None], k[None], v[None],
                                         is_causal=causal, scale=scale,
                                         enable_gqa=q.shape[0] != k.shape[0])
    return out[0]


@pytest.mark.parametrize("hq,hkv,d,bs,dtype", [
    (8, 2, 64, 16, "f16"), (4, 4, 128, 32, "bf16"), (8, 1, 64, 8, "bf16"),
    (16, 2, 128, 128, "f16"), (6, 3, 64, 16, "f16")])
def test_decode_equals_sdpa_on_contiguous_cache(hq, hkv, d, bs, dtype):
    cfg = small_cfg(hq=hq, hkv=hkv, d=d, bs=bs, nb=64 * 16 // bs + 8,
                    dtype=dtype, placement="identity",
                    lengths=("list", [1, 17, 250, 64, 100], None), seqs=5)
    x = W.make_inputs(cfg, seed=7)
    out = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                        hkv, bs, x.scale)
    for b in range(x.num_seqs):
        k, v = contiguous_kv(x, b)
        want = sdpa(x.q[b].double()[:, None, :], k, v, x.scale)[:, 0, :]
        np.testing.assert_allclose(out[b], want.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("hq,hkv,bs", [(4, 4, 16), (8, 2, 32), (4, 1, 128)])
def test_prefill_equals_sdpa_causal_on_contiguous_cache(hq, hkv, bs):
    cfg = small_cfg(kind="prefill", hq=hq, hkv=hkv, d=64, bs=bs, nb=80,
                    placement="identity", lengths=("list", [1, 37, 130, 5], None),
                    seqs=4)
    x = W.make_inputs(cfg, seed=11)
    # prefill reads the cache: write the new rows first (they are the whole
    # sequences here), through the oracle's own write.
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, bs)
    out = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                         x.context_lens, hkv, bs, x.scale, dtype=oracle.F16)
    xk = torch.from_numpy(kp.view(np.int16)).view(torch.float16)
    xv = torch.from_numpy(vp.view(np.int16)).view(torch.float16)
    x.k_pool, x.v_pool = xk, xv
    cu = x.cu_seqlens_q.tolist()
    for b in range(x.num_seqs):
        k, v = contiguous_kv(x, b)
        q = x.q[cu[b]:cu[b + 1]].double().permute(1, 0, 2)
        want = sdpa(q, k, v, x.scale, causal=True).permute(1, 0, 2)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], want.numpy(),
                                   rtol=1e-11, atol=1e-12)


def _decode_inputs(seed=3, **kw):
    return W.make_inputs(small_cfg(**kw), seed=seed)


def test_block_permutation_invariance_is_bitwise():
    x = _decode_inputs(seed=5, lengths=("uniform", 1, 120))
    base = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table,
                         x.context_lens, x.num_kv_heads, x.block_size, x.scale)
    rng = np.random.default_rng(9)
    perm = rng.permutation(x.num_blocks)          # new id of each old block
    inv = np.argsort(perm)
    kp2 = x.k_pool[torch.from_numpy(inv)]          # block perm[i] holds old i
    vp2 = x.v_pool[torch.from_numpy(inv)]
    bt = x.block_table.numpy().copy()
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    got = oracle.decode(x.q, kp2, vp2, bt2, x.context_lens, x.num_kv_heads,
                        x.block_size, x.scale)
    assert np.array_equal(got, base)


def test_single_key_returns_its_value_exactly():
    x = _decode_inputs(lengths=("fixed", 1, 1))
    out = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                        x.num_kv_heads, x.block_size, x.scale)
    g = x.num_q_heads // x.num_kv_heads
    for b in range(x.num_seqs):
        row = int(x.block_table[b, 0]) * x.block_size
        v = x.v_pool.reshape(-1, x.num_kv_heads, x.head_dim)[row].double().numpy()
        for h in range(x.num_q_heads):
            assert np.array_equal(out[b, h], v[h // g])


def test_constant_value_rows_return_that_value():
    x = _decode_inputs(lengths=("uniform", 2, 120))
    c = torch.linspace(-2, 2, x.head_dim, dtype=x.dtype)
    vp = torch.where(torch.isnan(x.v_pool), x.v_pool, c.expand_as(x.v_pool))
    out = oracle.decode(x.q, x.k_pool, vp, x.block_table, x.context_lens,
                        x.num_kv_heads, x.block_size, x.scale)
    want = c.double().numpy()
    for b in range(x.num_seqs):
        np.testing.assert_allclose(out[b], np.broadcast_to(want, out[b].shape),
                                   rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("zero", ["q", "scale"])
def test_flat_scores_give_mean_of_values(zero):
    x = _decode_inputs(lengths=("uniform", 1, 120))
    q = torch.zeros_like(x.q) if zero == "q" else x.q
    scale = 0.0 if zero == "scale" else x.scale
    out = oracle.decode(q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                        x.num_kv_heads, x.block_size, scale)
    g = x.num_q_heads // x.num_kv_heads
    flat_v = x.v_pool.reshape(-1, x.num_kv_heads, x.head_dim).double().numpy()
    for b in range(x.num_seqs):
        L = int(x.context_lens[b])
        rows = [int(x.block_table[b, j // x.block_size]) * x.block_size
                + j % x.block_size for j in range(L)]
        mean = flat_v[rows].mean(axis=0)
        for h in range(x.num_q_heads):
            np.testing.assert_allclose(out[b, h], mean[h // g], rtol=1e-12,
                                       atol=1e-13)


def test_zero_context_gives_zero_output():
    x = _decode_inputs(lengths=("list", [0, 5, 0, 3], None))
    out = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                        x.num_kv_heads, x.block_size, x.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out))
    assert np.abs(out[1]).sum() > 0


def test_decode_is_last_row_of_prefill():
    x = _decode_inputs(seed=21, lengths=("uniform", 1, 120))
    dec = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                        x.num_kv_heads, x.block_size, x.scale)
    # one query per sequence, bottom-right causal: it sees every key
    cu = np.arange(x.num_seqs + 1, dtype=np.int32)
    pre = oracle.prefill(x.q, x.k_pool, x.v_pool, x.block_table, cu,
                         x.context_lens, x.num_kv_heads, x.block_size, x.scale)
    assert np.array_equal(dec, pre)


def test_bottom_right_causal_equals_tail_of_full_causal():
    # chunked prefill: q < L queries are the last q rows of a full prefill
    cfg = small_cfg(kind="prefill", hq=4, hkv=2, d=64, bs=16, nb=40,
                    lengths=("list", [70, 33, 129], None), seqs=3)
    x = W.make_inputs(cfg, seed=13)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size)
    full = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                          x.context_lens, 2, 16, x.scale, dtype=oracle.F16)
    qlens = [5, 1, 64]
    cu = x.cu_seqlens_q.tolist()
    rows = np.concatenate([np.arange(cu[b + 1] - qlens[b], cu[b + 1])
                           for b in range(3)])
    q_tail = x.q[torch.from_numpy(rows)]
    cu_tail = oracle.cu_seqlens(qlens)
    tail = oracle.prefill(q_tail, kp, vp, x.block_table, cu_tail,
                          x.context_lens, 2, 16, x.scale, dtype=oracle.F16)
    assert np.array_equal(tail, full[rows])


def test_packed_equals_each_sequence_alone():
    cfg = small_cfg(kind="prefill", hq=4, hkv=4, d=64, bs=16, nb=40,
                    lengths=("list", [20, 1, 90, 47], None), seqs=4)
    x = W.make_inputs(cfg, seed=17)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size)
    packed = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                            x.context_lens, 4, 16, x.scale, dtype=oracle.F16)
    cu = x.cu_seqlens_q.tolist()
    for b in range(4):
        alone = oracle.prefill(x.q[cu[b]:cu[b + 1]], kp, vp,
                               x.block_table[b:b + 1], [0, cu[b + 1] - cu[b]],
                               x.context_lens[b:b + 1], 4, 16, x.scale,
                               dtype=oracle.F16)
        assert np.array_equal(alone, packed[cu[b]:cu[b + 1]])


def test_non_causal_prefill_rows_equal_decode():
    cfg = small_cfg(kind="prefill", hq=4, hkv=2, d=64, bs=16, nb=40,
                    lengths=("list", [30, 64], None), seqs=2)
    x = W.make_inputs(cfg, seed=19)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size)
    pre = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                         x.context_lens, 2, 16, x.scale, causal=False,
                         dtype=oracle.F16)
    cu = x.cu_seqlens_q.tolist()
    for b in range(2):
        for i in (0, 7, cu[b + 1] - cu[b] - 1):
            t = cu[b] + i
            dec = oracle.decode(x.q[t:t + 1], kp, vp, x.block_table[b:b + 1],
                                x.context_lens[b:b + 1], 2, 16, x.scale,
                                dtype=oracle.F16)
            assert np.array_equal(dec[0], pre[t])


def test_row_subset_matches_full():
    cfg = small_cfg(kind="prefill", hq=4, hkv=4, d=64, bs=16, nb=40,
                    lengths=("list", [50, 70], None), seqs=2)
    x = W.make_inputs(cfg, seed=23)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, x.block_size)
    full = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                          x.context_lens, 4, 16, x.scale, dtype=oracle.F16)
    rows = [0, 3, 49, 50, 119]
    sub = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                         x.context_lens, 4, 16, x.scale, rows=rows,
                         dtype=oracle.F16)
    assert np.array_equal(sub[rows], full[rows])
    others = np.setdiff1d(np.arange(120), rows)
    assert np.isnan(sub[others]).all()


def test_errors_reported():
    x = _decode_inputs(lengths=("list", [5, 40, 1, 9], None))
    bt = x.block_table.numpy().copy()
    bt[1, 1] = x.num_blocks            # block id out of range
    _, st = oracle.decode(x.q, x.k_pool, x.v_pool, bt, x.context_lens,
                          x.num_kv_heads, x.block_size, x.scale,
                          return_status=True)
    assert st == oracle.ERR_BLOCK
    ctx = x.context_lens.numpy().copy()
    ctx[2] = x.block_table.shape[1] * x.block_size + 1   # beyond capacity
    _, st = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, ctx,
                          x.num_kv_heads, x.block_size, x.scale,
                          return_status=True)
    assert st == oracle.ERR_LEN
    _, st = oracle.prefill(x.q, x.k_pool, x.v_pool, x.block_table,
                           [0, 2, 1, 3, 4], x.context_lens, x.num_kv_heads,
                           x.block_size, x.scale, return_status=True)
    assert st == oracle.ERR_LEN


def test_scale_enters_once():
    # doubling the scale equals doubling q (both multiply every score by 2):
    # a guard against the scale being dropped or applied twice.
    x = _decode_inputs(seed=29, dtype="bf16", lengths=("uniform", 10, 100))
    a = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                      x.num_kv_heads, x.block_size, 2 * x.scale)
    q2 = (x.q.float() * 2).to(x.dtype)   # exact: multiply by a power of two
    b = oracle.decode(q2, x.k_pool, x.v_pool, x.block_table, x.context_lens,
                      x.num_kv_heads, x.block_size, x.scale)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    assert math.isfinite(a.sum())
