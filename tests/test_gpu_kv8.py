"""INT8 KV pools on the GPU.

pa_reshape_and_cache_int8 must store the oracle's codes bit for bit, and
pa_decode_int8 must match the oracle's decode over the same codes within the
dtype's tolerance (cannbot-skills page App. A lists per-head dequantisation
scales for key and value; the quantisation rule -- round-half-even(x / scale)
in fp32, clamped to [-127, 127] -- is this library's reading, stated in
include/pa.h and pinned in the oracle's tests)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (W, assert_close, cfg, gpu, new_err, oracle_pools_after_write, pa,
                      require_gpu)

pytestmark = gpu

TORCH16 = {oracle.BF16: torch.bfloat16, oracle.F16: torch.float16}


def used_blocks(x_host):
    """Block ids the decode reads: the first ceil(L / block_size) of each row."""
    bt, bs = x_host.block_table.numpy(), x_host.block_size
    ids = [bt[b, :-(-int(L) // bs)] for b, L in enumerate(x_host.context_lens.tolist())]
    return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int64)


def head_scales(pool, hkv):
    """Per-KV-head absmax / 127 over the pool's finite values (fp32)."""
    a = pool.float().reshape(-1, hkv, pool.shape[-1])
    a = torch.where(torch.isfinite(a), a.abs(), torch.zeros_like(a))
    return (a.amax(dim=(0, 2)) / 127).clamp_min(1e-6).to(torch.float32).contiguous()


def as16(patterns, dtype_code):
    return torch.from_numpy(np.ascontiguousarray(patterns).view(np.int16)).view(
        TORCH16[dtype_code])


def int8_pools(x_host):
    """The oracle's codes of the workload's pools after this step's write
    (blocks the decode never reads stay 0)."""
    code = oracle.dtype_code(x_host.dtype)
    kp, vp = oracle_pools_after_write(x_host)
    used = torch.from_numpy(used_blocks(x_host).astype(np.int64))
    k16, v16 = as16(kp, code)[used], as16(vp, code)[used]
    hkv = x_host.num_kv_heads
    ks, vs = head_scales(k16, hkv), head_scales(v16, hkv)
    kc = np.zeros(kp.shape, np.int8)
    vc = np.zeros(vp.shape, np.int8)
    u = used.numpy()
    for g in range(hkv):
        kc[u, :, g] = oracle.quantize_int8(k16[:, :, g].contiguous(), float(ks[g]))
        vc[u, :, g] = oracle.quantize_int8(v16[:, :, g].contiguous(), float(vs[g]))
    return kc, vc, ks, vs


def gpu_decode_int8(x_host, kc, vc, ks, vs, partition_size, err):
    q = x_host.q.cuda()
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_int8(out, q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                      x_host.block_table.cuda(), x_host.context_lens.cuda(), ks.cuda(),
                      vs.cuda(), scale=x_host.scale, max_context_len=x_host.max_context_len,
                      partition_size=partition_size, d_error=err)
    return out


def oracle_decode_int8(x_host, kc, vc, ks, vs):
    return oracle.decode_int8(x_host.q, kc, vc, x_host.block_table, x_host.context_lens,
                              x_host.num_kv_heads, x_host.block_size, x_host.scale,
                              ks.numpy(), vs.numpy(), dtype=oracle.dtype_code(x_host.dtype))


def check_decode(x_host, partition_size, what):
    require_gpu()
    kc, vc, ks, vs = int8_pools(x_host)
    err = new_err()
    got = gpu_decode_int8(x_host, kc, vc, ks, vs, partition_size, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error bits {int(err.item())}"
    return assert_close(got, oracle_decode_int8(x_host, kc, vc, ks, vs), x_host.dtype,
                        what=what)


@pytest.mark.parametrize("partition_size", [0, 64, 512])
def test_llama7b_decode_int8(partition_size):
    check_decode(W.make_inputs("llama7b-decode"), partition_size, f"llama7b P{partition_size}")


def test_continuous_batching_int8():
    check_decode(W.make_inputs("continuous-batching"), 0, "continuous-batching")


def test_long_context_int8_full_size():
    x = W.make_inputs("long-context-decode")
    check_decode(x, x.partition_size, "long-context")


@pytest.mark.parametrize("bs,hq,hkv,dtype", [(16, 8, 2, "f16"), (32, 32, 8, "bf16"),
                                             (128, 64, 8, "bf16"), (8, 4, 4, "f16")])
@pytest.mark.parametrize("partition_size", [0, 64])
def test_int8_grid(bs, hq, hkv, dtype, partition_size):
    lengths = [0, 1, bs - 1, bs, bs + 1, 63, 200, 333]
    c = cfg(hq=hq, hkv=hkv, d=128, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 8,
            dtype=dtype, lengths=lengths)
    x = W.make_inputs(c, seed=300 + bs + hq)
    check_decode(x, partition_size, f"bs{bs} g{hq // hkv} {dtype} P{partition_size}")


def test_int8_decode_bad_scale_gives_zero_heads():
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[40, 90, 17]), seed=8)
    kc, vc, ks, vs = int8_pools(x)
    bad = ks.clone()
    bad[0] = -1.0
    err = new_err()
    got = gpu_decode_int8(x, kc, vc, bad, vs, 0, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SCALE
    g = got.double().cpu().numpy()
    assert (g[:, :4] == 0).all()  # the queries of KV head 0
    want = oracle_decode_int8(x, kc, vc, ks, vs)
    assert np.abs(g[:, 4:] - want[:, 4:]).max() <= 1e-2


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_write_int8_bit_exact(dtype):
    require_gpu()
    c = cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype=dtype, lengths=[30, 50, 17, 64],
            write_new_token=True)
    x = W.make_inputs(c, seed=21)
    kn, vn = x.k_new.clone(), x.v_new.clone()
    kn[1] *= 100  # beyond the code range: clamped
    vn[2] *= -100
    slots = x.slot_mapping.clone()
    slots[3] = -1                                 # padding: nothing written
    n = slots.numel()
    slots = torch.cat([slots, torch.tensor([64 * 16 + 5])])  # past the pool
    kn = torch.cat([kn, kn[:1]])
    vn = torch.cat([vn, vn[:1]])
    shape = tuple(x.k_pool.shape)
    g = torch.Generator().manual_seed(4)
    k0 = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
    v0 = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
    ks = torch.tensor([0.021, 0.0137], dtype=torch.float32)
    vs = torch.tensor([0.0093, 0.05], dtype=torch.float32)
    kd, vd, err = k0.cuda(), v0.cuda(), new_err()
    pa.pa_reshape_and_cache_int8(kn.cuda(), vn.cuda(), kd, vd, slots.cuda(), ks.cuda(),
                                 vs.cuda(), d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.DEVERR_SLOT
    kw, vw = k0.numpy().copy(), v0.numpy().copy()
    st = oracle.write_int8(kw, vw, kn, vn, slots.numpy(), 16, ks.numpy(), vs.numpy())
    assert st == oracle.ERR_SLOT and n == 4
    assert np.array_equal(kd.cpu().numpy(), kw)
    assert np.array_equal(vd.cpu().numpy(), vw)


def test_write_int8_bad_scale():
    require_gpu()
    x = W.make_inputs(cfg(hq=4, hkv=2, d=128, bs=16, nb=16, dtype="bf16", lengths=[9, 20],
                          write_new_token=True), seed=6)
    shape = tuple(x.k_pool.shape)
    kd = torch.full(shape, 7, dtype=torch.int8, device="cuda")
    vd = torch.full(shape, 7, dtype=torch.int8, device="cuda")
    ks = torch.tensor([0.0, 0.02], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.01, 0.02], dtype=torch.float32, device="cuda")
    err = new_err()
    pa.pa_reshape_and_cache_int8(x.k_new.cuda(), x.v_new.cuda(), kd, vd, x.slot_mapping.cuda(),
                                 ks, vs, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SCALE
    kw = np.full(shape, 7, np.int8)
    vw = np.full(shape, 7, np.int8)
    st = oracle.write_int8(kw, vw, x.k_new, x.v_new, x.slot_mapping.numpy(), 16,
                           ks.cpu().numpy(), vs.cpu().numpy())
    assert st == oracle.ERR_SCALE
    assert np.array_equal(kd.cpu().numpy(), kw) and np.array_equal(vd.cpu().numpy(), vw)


def test_decode_write_int8_step():
    """pa_decode_write_int8 = the oracle's INT8 write of the step's new tokens,
    then its INT8 decode over the updated pools (llama7b-decode, full size)."""
    require_gpu()
    x = W.make_inputs("llama7b-decode")
    kc, vc, ks, vs = int8_pools(x)  # the codes after this step's write
    hkv, d = x.num_kv_heads, x.head_dim
    slots = x.slot_mapping.numpy()
    k0, v0 = kc.copy(), vc.copy()
    k0.reshape(-1, hkv, d)[slots] = 0  # before the write
    v0.reshape(-1, hkv, d)[slots] = 0
    kw, vw = k0.copy(), v0.copy()
    assert oracle.write_int8(kw, vw, x.k_new, x.v_new, slots, x.block_size, ks.numpy(),
                             vs.numpy()) == oracle.OK
    assert np.array_equal(kw, kc) and np.array_equal(vw, vc)

    kd, vd, err = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda(), new_err()
    q = x.q.cuda()
    out = torch.full_like(q, float("nan"))
    pa.pa_decode_write_int8(out, q, x.k_new.cuda(), x.v_new.cuda(), kd, vd,
                            x.slot_mapping.cuda(), x.block_table.cuda(), x.context_lens.cuda(),
                            ks.cuda(), vs.cuda(), scale=x.scale,
                            max_context_len=x.max_context_len, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    assert_close(out, oracle_decode_int8(x, kc, vc, ks, vs), x.dtype, what="INT8 step")
