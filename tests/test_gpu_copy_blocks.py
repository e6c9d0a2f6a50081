"""pa_copy_blocks on the GPU.

Copy-on-write of whole blocks (coreui.cn "Ascend CANN ATB KV Cache and
PagedAttention", page update race: a request that appends to a shared page
first copies the page to a free one): the pools after the call must equal the
oracle's byte for byte, for 16-bit and INT8 pools, ragged block sizes and bad
pairs; a forked sequence must then decode like the oracle; at the benchmark's
full size every destination block must equal its source."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (W, assert_close, cfg, gpu, new_err, oracle_pools_after_write, pa,
                      require_gpu, u16)

pytestmark = gpu


def pools(nb, bs, hkv, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    shape = (nb, bs, hkv, d)
    if dtype == torch.int8:
        return (torch.randint(-128, 128, shape, generator=g, dtype=torch.int8),
                torch.randint(-128, 128, shape, generator=g, dtype=torch.int8))
    return (torch.randn(shape, generator=g).to(dtype), torch.randn(shape, generator=g).to(dtype))


def raw(t):
    """The pool's bytes as a numpy array [num_blocks, -1] (the oracle copies bytes)."""
    t = t.contiguous()
    return t.view(torch.uint8).reshape(t.shape[0], -1).numpy()


def run(k, v, pairs, expect_err=0):
    require_gpu()
    mapping = torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2)
    kd, vd, err = k.cuda(), v.cuda(), new_err()
    pa.pa_copy_blocks(kd, vd, mapping.cuda(), d_error=err)
    torch.cuda.synchronize()
    kw, vw = raw(k).copy(), raw(v).copy()
    st = oracle.copy_blocks(kw, vw, mapping.numpy())
    assert int(err.item()) == expect_err
    assert st == (oracle.ERR_BLOCK if expect_err else oracle.OK)
    assert np.array_equal(raw(kd.cpu()), kw)
    assert np.array_equal(raw(vd.cpu()), vw)


@pytest.mark.parametrize("bs,hkv,d,dtype", [
    (16, 32, 128, torch.bfloat16),  # 128 KB blocks: eight 16 KB slices
    (16, 2, 64, torch.float16),     # 4 KB: part of one slice
    (128, 8, 128, torch.bfloat16),  # 256 KB: sixteen slices
    (8, 3, 40, torch.float16),      # 1920 B: 120 vectors, not a multiple of the CTA
    (16, 8, 128, torch.int8),       # INT8 pool
    (32, 5, 128, torch.int8),       # 20 KB: a slice and a ragged rest
])
def test_copy_blocks_bit_exact(bs, hkv, d, dtype):
    nb = 64
    k, v = pools(nb, bs, hkv, d, dtype, seed=bs + hkv + d)
    ids = np.random.default_rng(bs * 7 + d).permutation(nb)
    # sources and destinations disjoint, plus one block copied onto itself
    pairs = [[int(ids[i]), int(ids[i + 24])] for i in range(24)] + [[int(ids[50])] * 2]
    run(k, v, pairs)


def test_copy_blocks_bad_pairs_are_skipped_and_reported():
    k, v = pools(16, 16, 2, 64, torch.bfloat16, 3)
    run(k, v, [[1, 2], [16, 3], [-1, 4], [5, 16], [6, 7]], expect_err=pa.DEVERR_BLOCK_ID)


def test_copy_blocks_no_pairs():
    require_gpu()
    k, v = pools(8, 16, 2, 64, torch.float16, 4)
    kd, vd, err = k.cuda(), v.cuda(), new_err()
    pa.pa_copy_blocks(kd, vd, torch.zeros(0, 2, dtype=torch.int64, device="cuda"), d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)


def test_copy_on_write_fork_then_decode():
    """Sequence B forks from A (sharing A's blocks), copies A's partly filled
    last block to a free block, appends its own token there; one decode call
    then serves A and B, and must match the oracle doing the same steps."""
    require_gpu()
    L, bs = 37, 16
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=bs, nb=64, dtype="bf16", lengths=[L],
                          write_new_token=True), seed=5)
    nblk = -(-L // bs)
    bt_a = x.block_table[0].tolist()
    free = next(b for b in range(64) if b not in bt_a[:nblk])
    bt = torch.full((2, x.block_table.shape[1]), -1, dtype=torch.int32)
    bt[0, :nblk] = torch.tensor(bt_a[:nblk])
    bt[1, :nblk] = torch.tensor(bt_a[:nblk - 1] + [free])
    lens = torch.tensor([L, L + 1], dtype=torch.int32)
    mapping = torch.tensor([[bt_a[nblk - 1], free]], dtype=torch.int64)
    slot = torch.tensor([free * bs + L % bs], dtype=torch.int64)
    g = torch.Generator().manual_seed(6)
    kb = torch.randn(1, 2, 128, generator=g).to(torch.bfloat16)
    vb = torch.randn(1, 2, 128, generator=g).to(torch.bfloat16)
    q = torch.randn(2, 8, 128, generator=g).to(torch.bfloat16)

    # A's last token comes from this step's write; then B forks
    kd, vd, err = x.k_pool.cuda(), x.v_pool.cuda(), new_err()
    pa.pa_reshape_and_cache(x.k_new.cuda(), x.v_new.cuda(), kd, vd, x.slot_mapping.cuda(),
                            d_error=err)
    pa.pa_copy_blocks(kd, vd, mapping.cuda(), d_error=err)
    pa.pa_reshape_and_cache(kb.cuda(), vb.cuda(), kd, vd, slot.cuda(), d_error=err)
    out = torch.empty(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    pa.pa_decode(out, q.cuda(), kd, vd, bt.cuda(), lens.cuda(), scale=x.scale,
                 max_context_len=L + 1, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    kp, vp = oracle_pools_after_write(x)
    assert oracle.copy_blocks(kp, vp, mapping.numpy()) == oracle.OK
    assert oracle.write(kp, vp, kb, vb, slot.numpy(), bs) == oracle.OK
    want = oracle.decode(q, kp, vp, bt, lens, 2, bs, x.scale)
    assert_close(out, want, torch.bfloat16, what="copy-on-write fork")
    assert np.array_equal(u16(kd.cpu()), kp) and np.array_equal(u16(vd.cpu()), vp)


def test_copy_blocks_full_size():
    """The benchmark's workload: 1024 of the 8192 blocks of the llama7b
    pools (bs 16, 32 KV heads, D 128, bf16; 128 KB per block and pool)
    copied to 1024 others; every destination equals its source and nothing
    else changes."""
    require_gpu()
    nb, n = 8192, 1024
    g = torch.Generator(device="cuda").manual_seed(11)
    k = torch.randn(nb, 16, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(nb, 16, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    ids = torch.randperm(nb, generator=g, device="cuda")
    src, dst = ids[:n], ids[n:2 * n]
    k0, v0 = k.clone(), v.clone()
    err = new_err()
    pa.pa_copy_blocks(k, v, torch.stack([src, dst], dim=1).contiguous(), d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(k[dst].view(torch.int16), k0[src].view(torch.int16))
    assert torch.equal(v[dst].view(torch.int16), v0[src].view(torch.int16))
    keep = torch.ones(nb, dtype=torch.bool, device="cuda")
    keep[dst] = False
    assert torch.equal(k[keep].view(torch.int16), k0[keep].view(torch.int16))
    assert torch.equal(v[keep].view(torch.int16), v0[keep].view(torch.int16))
