"""pa_decode on the GPU against the fp64 oracle, element by element, plus the
invariants the pages fix (block permutation, aliasing, split = unsplit)."""
import numpy as np
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, gpu_decode, gpu_write, new_err,
                      oracle_decode, oracle_pools_after_write, pa, require_gpu, u16)

pytestmark = gpu


def _run(x_host, partition_size=None, what=""):
    require_gpu()
    kp, vp = oracle_pools_after_write(x_host)
    want = oracle_decode(x_host, kp, vp)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    out = gpu_decode(x, partition_size=partition_size, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert np.array_equal(u16(x.k_pool), kp)  # the write feeding the decode
    e = assert_close(out, want, x.dtype, what=what)
    return out, e


@pytest.mark.parametrize("name", ["tiny-decode", "llama7b-decode", "continuous-batching",
                                  "long-context-decode"])
def test_named_config_full_size(name):
    # Full sizes, in the launch configuration the benchmark times.
    _run(W.make_inputs(name), what=name)


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (8, 2), (16, 2)])
def test_edge_lengths_grid(bs, d, hq, hkv):
    lengths = [0, 1, bs - 1, bs, bs + 1, 63, 64, 65, 129, 300]
    lengths = [max(0, n) for n in lengths]
    c = cfg(hq=hq, hkv=hkv, d=d, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 4,
            dtype="bf16" if (bs + d) % 3 else "f16", lengths=lengths)
    x = W.make_inputs(c, seed=100 + bs + d + hq)
    for part in (64, 0):
        _run(x, partition_size=part, what=f"bs{bs} d{d} g{hq // hkv} P{part}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_split_equals_unsplit(dtype):
    x = W.make_inputs(cfg(hq=16, hkv=2, d=128, bs=32, nb=600, dtype=dtype,
                          lengths=[1000, 3000, 64, 2049]), seed=21)
    outs = [_run(x, partition_size=p, what=f"P{p}")[0] for p in (64, 256, 512, 4096)]
    tol = 2e-3 if dtype == "f16" else 1e-2
    for o in outs[1:]:
        assert (o.double() - outs[-1].double()).abs().max().item() <= tol


def test_block_permutation_invariance_bitwise():
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=400, lengths=[700, 1500, 33]),
                      seed=23)
    a = gpu_decode(x.to("cuda"), partition_size=256)
    perm = np.random.default_rng(3).permutation(x.num_blocks)
    inv = torch.from_numpy(np.argsort(perm))
    bt = x.block_table.numpy()
    x2 = x.to("cpu")
    x2.k_pool, x2.v_pool = x.k_pool[inv], x.v_pool[inv]
    x2.block_table = torch.from_numpy(np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
                                      .astype(np.int32))
    b = gpu_decode(x2.to("cuda"), partition_size=256)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_blocks_equal_private_copies():
    # Two sequences alias the same physical prefix blocks (prefix sharing).
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=8, d=128, bs=16, nb=200, lengths=[200, 200, 200]),
                      seed=29)
    shared = x.to("cpu")
    bt = shared.block_table.clone()
    bt[1, :8] = bt[0, :8]          # first 128 tokens of seq 1 read seq 0's blocks
    shared.block_table = bt
    private = x.to("cpu")          # seq 1 keeps its own blocks, with seq 0's data
    kp, vp = private.k_pool.clone(), private.v_pool.clone()
    for j in range(8):
        kp[x.block_table[1, j]] = kp[x.block_table[0, j]]
        vp[x.block_table[1, j]] = vp[x.block_table[0, j]]
    private.k_pool, private.v_pool = kp, vp
    a = gpu_decode(shared.to("cuda"), partition_size=64)
    b = gpu_decode(private.to("cuda"), partition_size=64)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    kp0, vp0 = u16(shared.k_pool), u16(shared.v_pool)
    assert_close(a, oracle_decode(shared, kp0, vp0), x.dtype)


def test_strided_query_and_output():
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=64, bs=32, nb=64, dtype="f16",
                          lengths=[90, 400, 7]), seed=31)
    xd = x.to("cuda")
    big_q = torch.zeros(3, 8 * 64 + 64, dtype=x.dtype, device="cuda")
    big_q[:, :512] = xd.q.reshape(3, 512)
    q_view = big_q[:, :512].view(3, 8, 64)
    big_o = torch.full((3, 8 * 64 + 128), 7.0, dtype=x.dtype, device="cuda")
    o_view = big_o[:, :512].view(3, 8, 64)
    xd.q = q_view
    gpu_decode(xd, out=o_view, partition_size=128)
    torch.cuda.synchronize()
    assert (big_o[:, 512:] == 7.0).all()
    kp, vp = u16(x.k_pool), u16(x.v_pool)
    assert_close(o_view, oracle_decode(x, kp, vp), x.dtype)


def test_special_cases_single_key_and_constant_value():
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, lengths=[1, 1, 50, 80]),
                      seed=37)
    c = torch.linspace(-1.5, 1.5, 128, dtype=x.dtype)
    rows = x.v_pool.view(-1, 2, 128)
    for b in (2, 3):
        for j in range(int(x.context_lens[b])):
            r = int(x.block_table[b, j // 16]) * 16 + j % 16
            rows[r] = c
    out = gpu_decode(x.to("cuda")).cpu()
    for b in (0, 1):  # a single key returns its value row exactly
        r = int(x.block_table[b, 0]) * 16
        for h in range(8):
            assert torch.equal(out[b, h], rows[r, h // 4])
    for b in (2, 3):  # constant value rows return that value
        assert (out[b].float() - c.float()).abs().max().item() <= 1e-2


def test_zero_lengths_give_zero():
    require_gpu()
    x = W.make_inputs(cfg(hq=4, hkv=4, d=128, bs=16, nb=16, lengths=[0, 5, 0]), seed=41)
    out = gpu_decode(x.to("cuda"), partition_size=64)
    torch.cuda.synchronize()
    assert (out[0] == 0).all() and (out[2] == 0).all() and torch.isfinite(out).all()


def test_device_errors_are_flagged_not_faults():
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, lengths=[40, 100, 30, 70]),
                      seed=43)
    # a bad block id inside sequence 1's range
    bad = x.to("cpu")
    bt = bad.block_table.clone()
    bt[1, 2] = 10_000
    bad.block_table = bt
    err = new_err()
    out = gpu_decode(bad.to("cuda"), err=err, partition_size=64)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_BLOCK_ID
    assert torch.isfinite(out[[0, 2, 3]]).all()
    # a context length beyond the block table's capacity / the host hint
    for ctx_bad, hint in ((bad.block_table.shape[1] * 16 + 1, None), (100, 90)):
        y = x.to("cpu")
        cl = y.context_lens.clone()
        cl[2] = ctx_bad
        y.context_lens = cl
        err = new_err()
        out = gpu_decode(y.to("cuda"), err=err, partition_size=64,
                         max_context_len=hint if hint else max(ctx_bad, 100))
        torch.cuda.synchronize()
        assert int(err.item()) & pa.DEVERR_CONTEXT
        assert (out[2] == 0).all()
