"""8-bit KV pools (INT8 and FP8 E4M3) on the GPU.

The writes must store the oracle's codes bit for bit, and the decodes must
match the oracle's decode over the same codes within the dtype's tolerance
(cannbot-skills page App. A lists per-head dequantisation scales for key and
value; the quantisation rules -- INT8: round-half-even(x / scale) in fp32,
clamped to +-127; FP8: the nearest E4M3 value to x / scale, ties to even,
saturating at 448 -- are this library's readings, stated in include/pa.h and
pinned in the oracle's tests).  Every test runs for both formats."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (W, assert_close, cfg, gpu, new_err, oracle_pools_after_write, pa,
                      require_gpu)

pytestmark = gpu

TORCH16 = {oracle.BF16: torch.bfloat16, oracle.F16: torch.float16}
FORMATS = ["int8", "fp8"]
CODE_DTYPE = {"int8": np.int8, "fp8": np.uint8}
CODE_MAX = {"int8": 127.0, "fp8": 448.0}
# a byte the write never stores, placed where no decode may look: INT8 -128,
# FP8 a NaN code
POISON = {"int8": -128, "fp8": 0x7F}
QUANTIZE = {"int8": oracle.quantize_int8, "fp8": oracle.quantize_fp8}
ORACLE_WRITE = {"int8": oracle.write_int8, "fp8": oracle.write_fp8}
ORACLE_DECODE = {"int8": oracle.decode_int8, "fp8": oracle.decode_fp8}
GPU_WRITE = {"int8": pa.pa_reshape_and_cache_int8, "fp8": pa.pa_reshape_and_cache_fp8}
GPU_DECODE = {"int8": pa.pa_decode_int8, "fp8": pa.pa_decode_fp8}
GPU_STEP = {"int8": pa.pa_decode_write_int8, "fp8": pa.pa_decode_write_fp8}


def used_blocks(x_host):
    """Block ids the decode reads: the first ceil(L / block_size) of each row."""
    bt, bs = x_host.block_table.numpy(), x_host.block_size
    ids = [bt[b, :-(-int(L) // bs)] for b, L in enumerate(x_host.context_lens.tolist())]
    return np.unique(np.concatenate(ids)) if ids else np.zeros(0, np.int64)


def head_scales(pool, hkv, fmt):
    """Per-KV-head absmax / (largest code) over the pool's finite values (fp32)."""
    a = pool.float().reshape(-1, hkv, pool.shape[-1])
    a = torch.where(torch.isfinite(a), a.abs(), torch.zeros_like(a))
    return (a.amax(dim=(0, 2)) / CODE_MAX[fmt]).clamp_min(1e-6).to(torch.float32).contiguous()


def as16(patterns, dtype_code):
    return torch.from_numpy(np.ascontiguousarray(patterns).view(np.int16)).view(
        TORCH16[dtype_code])


def poison_past_context(pool, x_host, fmt):
    """Rows of the used blocks past each sequence's context get POISON."""
    bt, bs = x_host.block_table.numpy(), x_host.block_size
    flat = pool.reshape(-1, *pool.shape[2:])
    for b, L in enumerate(x_host.context_lens.tolist()):
        n = -(-int(L) // bs)
        for j in range(int(L), n * bs):
            flat[int(bt[b, j // bs]) * bs + j % bs] = POISON[fmt]


def pools8(x_host, fmt):
    """The oracle's codes of the workload's pools after this step's write
    (blocks the decode never reads stay 0, rows past a context hold POISON)."""
    code = oracle.dtype_code(x_host.dtype)
    kp, vp = oracle_pools_after_write(x_host)
    used = torch.from_numpy(used_blocks(x_host).astype(np.int64))
    k16, v16 = as16(kp, code)[used], as16(vp, code)[used]
    hkv = x_host.num_kv_heads
    ks, vs = head_scales(k16, hkv, fmt), head_scales(v16, hkv, fmt)
    kc = np.zeros(kp.shape, CODE_DTYPE[fmt])
    vc = np.zeros(vp.shape, CODE_DTYPE[fmt])
    u = used.numpy()
    for g in range(hkv):
        kc[u, :, g] = QUANTIZE[fmt](k16[:, :, g].contiguous(), float(ks[g]))
        vc[u, :, g] = QUANTIZE[fmt](v16[:, :, g].contiguous(), float(vs[g]))
    poison_past_context(kc, x_host, fmt)
    poison_past_context(vc, x_host, fmt)
    return kc, vc, ks, vs


def gpu_decode8(fmt, x_host, kc, vc, ks, vs, partition_size, err):
    q = x_host.q.cuda()
    out = torch.full_like(q, float("nan"))
    GPU_DECODE[fmt](out, q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                    x_host.block_table.cuda(), x_host.context_lens.cuda(), ks.cuda(), vs.cuda(),
                    scale=x_host.scale, max_context_len=x_host.max_context_len,
                    partition_size=partition_size, d_error=err)
    return out


def oracle_decode8(fmt, x_host, kc, vc, ks, vs):
    return ORACLE_DECODE[fmt](x_host.q, kc, vc, x_host.block_table, x_host.context_lens,
                              x_host.num_kv_heads, x_host.block_size, x_host.scale,
                              ks.numpy(), vs.numpy(), dtype=oracle.dtype_code(x_host.dtype))


def check_decode(fmt, x_host, partition_size, what):
    require_gpu()
    kc, vc, ks, vs = pools8(x_host, fmt)
    err = new_err()
    got = gpu_decode8(fmt, x_host, kc, vc, ks, vs, partition_size, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error bits {int(err.item())}"
    return assert_close(got, oracle_decode8(fmt, x_host, kc, vc, ks, vs), x_host.dtype,
                        what=f"{fmt} {what}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("partition_size", [0, 64, 512])
def test_llama7b_decode(fmt, partition_size):
    check_decode(fmt, W.make_inputs("llama7b-decode"), partition_size,
                 f"llama7b P{partition_size}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_continuous_batching(fmt):
    check_decode(fmt, W.make_inputs("continuous-batching"), 0, "continuous-batching")


@pytest.mark.parametrize("fmt", FORMATS)
def test_long_context_full_size(fmt):
    x = W.make_inputs("long-context-decode")
    check_decode(fmt, x, x.partition_size, "long-context")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("bs,hq,hkv,dtype", [(16, 8, 2, "f16"), (32, 32, 8, "bf16"),
                                             (128, 64, 8, "bf16"), (8, 4, 4, "f16")])
@pytest.mark.parametrize("partition_size", [0, 64])
def test_grid(fmt, bs, hq, hkv, dtype, partition_size):
    lengths = [0, 1, bs - 1, bs, bs + 1, 63, 200, 333]
    c = cfg(hq=hq, hkv=hkv, d=128, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 8,
            dtype=dtype, lengths=lengths)
    x = W.make_inputs(c, seed=300 + bs + hq)
    check_decode(fmt, x, partition_size, f"bs{bs} g{hq // hkv} {dtype} P{partition_size}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_decode_bad_scale_gives_zero_heads(fmt):
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[40, 90, 17]), seed=8)
    kc, vc, ks, vs = pools8(x, fmt)
    bad = ks.clone()
    bad[0] = -1.0
    err = new_err()
    got = gpu_decode8(fmt, x, kc, vc, bad, vs, 0, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SCALE
    g = got.double().cpu().numpy()
    assert (g[:, :4] == 0).all()  # the queries of KV head 0
    want = oracle_decode8(fmt, x, kc, vc, ks, vs)
    assert np.abs(g[:, 4:] - want[:, 4:]).max() <= 1e-2


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_write_bit_exact(fmt, dtype):
    require_gpu()
    c = cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype=dtype, lengths=[30, 50, 17, 64],
            write_new_token=True)
    x = W.make_inputs(c, seed=21)
    kn, vn = x.k_new.clone(), x.v_new.clone()
    kn[1] *= 100  # beyond the code range: clamped / saturated
    vn[2] *= -100
    kn[0, 0, :4] = torch.tensor([float("nan"), -0.0, 1e-30, -1e-30])  # NaN, signed zeros
    slots = x.slot_mapping.clone()
    slots[3] = -1                                 # padding: nothing written
    n = slots.numel()
    slots = torch.cat([slots, torch.tensor([64 * 16 + 5])])  # past the pool
    kn = torch.cat([kn, kn[:1]])
    vn = torch.cat([vn, vn[:1]])
    shape = tuple(x.k_pool.shape)
    g = torch.Generator().manual_seed(4)
    k0 = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8).numpy().view(
        CODE_DTYPE[fmt])
    v0 = torch.randint(0, 256, shape, generator=g, dtype=torch.uint8).numpy().view(
        CODE_DTYPE[fmt])
    ks = torch.tensor([0.021, 0.0137], dtype=torch.float32)
    vs = torch.tensor([0.0093, 0.05], dtype=torch.float32)
    kd, vd, err = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda(), new_err()
    GPU_WRITE[fmt](kn.cuda(), vn.cuda(), kd, vd, slots.cuda(), ks.cuda(), vs.cuda(),
                   d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.DEVERR_SLOT
    kw, vw = k0.copy(), v0.copy()
    st = ORACLE_WRITE[fmt](kw, vw, kn, vn, slots.numpy(), 16, ks.numpy(), vs.numpy())
    assert st == oracle.ERR_SLOT and n == 4
    assert np.array_equal(kd.cpu().numpy(), kw)
    assert np.array_equal(vd.cpu().numpy(), vw)


@pytest.mark.parametrize("fmt", FORMATS)
def test_write_bad_scale(fmt):
    require_gpu()
    x = W.make_inputs(cfg(hq=4, hkv=2, d=128, bs=16, nb=16, dtype="bf16", lengths=[9, 20],
                          write_new_token=True), seed=6)
    shape = tuple(x.k_pool.shape)
    kw = np.full(shape, 7, CODE_DTYPE[fmt])
    vw = np.full(shape, 7, CODE_DTYPE[fmt])
    kd, vd = torch.from_numpy(kw.copy()).cuda(), torch.from_numpy(vw.copy()).cuda()
    ks = torch.tensor([0.0, 0.02], dtype=torch.float32, device="cuda")
    vs = torch.tensor([0.01, 0.02], dtype=torch.float32, device="cuda")
    err = new_err()
    GPU_WRITE[fmt](x.k_new.cuda(), x.v_new.cuda(), kd, vd, x.slot_mapping.cuda(), ks, vs,
                   d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SCALE
    st = ORACLE_WRITE[fmt](kw, vw, x.k_new, x.v_new, x.slot_mapping.numpy(), 16,
                           ks.cpu().numpy(), vs.cpu().numpy())
    assert st == oracle.ERR_SCALE
    assert np.array_equal(kd.cpu().numpy(), kw) and np.array_equal(vd.cpu().numpy(), vw)


@pytest.mark.parametrize("fmt", FORMATS)
def test_decode_write_step(fmt):
    """The one-call step = the oracle's write of the step's new tokens, then
    its decode over the updated pools (llama7b-decode, full size)."""
    require_gpu()
    x = W.make_inputs("llama7b-decode")
    kc, vc, ks, vs = pools8(x, fmt)  # the codes after this step's write
    hkv, d = x.num_kv_heads, x.head_dim
    slots = x.slot_mapping.numpy()
    k0, v0 = kc.copy(), vc.copy()
    k0.reshape(-1, hkv, d)[slots] = 0  # before the write
    v0.reshape(-1, hkv, d)[slots] = 0
    kw, vw = k0.copy(), v0.copy()
    assert ORACLE_WRITE[fmt](kw, vw, x.k_new, x.v_new, slots, x.block_size, ks.numpy(),
                             vs.numpy()) == oracle.OK
    assert np.array_equal(kw, kc) and np.array_equal(vw, vc)

    kd, vd, err = torch.from_numpy(k0).cuda(), torch.from_numpy(v0).cuda(), new_err()
    q = x.q.cuda()
    out = torch.full_like(q, float("nan"))
    GPU_STEP[fmt](out, q, x.k_new.cuda(), x.v_new.cuda(), kd, vd, x.slot_mapping.cuda(),
                  x.block_table.cuda(), x.context_lens.cuda(), ks.cuda(), vs.cuda(),
                  scale=x.scale, max_context_len=x.max_context_len, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
    assert_close(out, oracle_decode8(fmt, x, kc, vc, ks, vs), x.dtype, what=f"{fmt} step")


def test_fp8_pool_as_float8_tensor():
    """FP8 pools may be float8_e4m3fn tensors (the same bytes as uint8)."""
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=32, dtype="bf16", lengths=[50, 7]),
                      seed=9)
    kc, vc, ks, vs = pools8(x, "fp8")
    q = x.q.cuda()
    out = torch.empty_like(q)
    kf = torch.from_numpy(kc).cuda().view(torch.float8_e4m3fn)
    vf = torch.from_numpy(vc).cuda().view(torch.float8_e4m3fn)
    pa.pa_decode_fp8(out, q, kf, vf, x.block_table.cuda(), x.context_lens.cuda(), ks.cuda(),
                     vs.cuda(), scale=x.scale, max_context_len=x.max_context_len)
    torch.cuda.synchronize()
    assert_close(out, oracle_decode8("fp8", x, kc, vc, ks, vs), x.dtype, what="float8 pools")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("partition_size", [0, 64])
def test_device_errors_are_flagged(fmt, partition_size):
    """A bad block id, then a context past the block table: flagged in
    d_error, never a fault; the other sequences still match the oracle."""
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[40, 100, 30, 70]), seed=43)
    kc, vc, ks, vs = pools8(x, fmt)
    want = oracle_decode8(fmt, x, kc, vc, ks, vs)
    bt = x.block_table.clone()
    bt[1, 2] = 10_000
    cases = [(bt, x.context_lens, pa.DEVERR_BLOCK_ID, 1)]
    cl = x.context_lens.clone()
    cl[2] = x.block_table.shape[1] * x.block_size + 1  # past the block table's capacity
    cases.append((x.block_table, cl, pa.DEVERR_CONTEXT, 2))
    for bt_c, cl_c, bit, bad in cases:
        q = x.q.cuda()
        out = torch.full_like(q, float("nan"))
        err = new_err()
        GPU_DECODE[fmt](out, q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                        bt_c.cuda(), cl_c.cuda(), ks.cuda(), vs.cuda(), scale=x.scale,
                        max_context_len=int(cl_c.max()), partition_size=partition_size,
                        d_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) & bit
        g = out.double().cpu().numpy()
        rows = [r for r in range(4) if r != bad]  # every other sequence is intact
        assert np.isfinite(g[rows]).all()
        assert np.abs(g[rows] - want[rows]).max() <= 1e-2
        if bit == pa.DEVERR_CONTEXT:
            assert (g[bad] == 0).all()


def _decode_codes(fmt, x, kc, vc, ks, vs, bt, cl, partition_size=0):
    q = x.q.cuda()
    out = torch.empty_like(q)
    GPU_DECODE[fmt](out, q, torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                    bt.cuda(), cl.cuda(), ks.cuda(), vs.cuda(), scale=x.scale,
                    max_context_len=int(cl.max()), partition_size=partition_size)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("fmt", FORMATS)
def test_block_permutation_invariance_bitwise(fmt):
    """Moving the physical blocks (and the block table with them) changes
    nothing in the output, bit for bit."""
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[40, 100, 30, 70]), seed=51)
    kc, vc, ks, vs = pools8(x, fmt)
    perm = np.random.default_rng(5).permutation(kc.shape[0])
    kp, vp = np.empty_like(kc), np.empty_like(vc)
    kp[perm], vp[perm] = kc, vc
    bt = x.block_table.clone()
    ok = bt >= 0
    bt[ok] = torch.from_numpy(perm).to(torch.int32)[bt[ok].long()]
    a = _decode_codes(fmt, x, kc, vc, ks, vs, x.block_table, x.context_lens)
    b = _decode_codes(fmt, x, kp, vp, ks, vs, bt, x.context_lens)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
def test_shared_blocks_equal_private_copies(fmt):
    """Two sequences whose tables name the same physical blocks (a shared
    prefix) decode like two sequences with private copies of those blocks."""
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[64, 64]), seed=52)
    kc, vc, ks, vs = pools8(x, fmt)
    shared = x.block_table.clone()
    shared[1] = shared[0]  # sequence 1 reads sequence 0's blocks
    kq, vq = kc.copy(), vc.copy()
    for j in range(4):  # private copies: sequence 0's blocks copied into sequence 1's
        kq[int(x.block_table[1, j])] = kc[int(x.block_table[0, j])]
        vq[int(x.block_table[1, j])] = vc[int(x.block_table[0, j])]
    a = _decode_codes(fmt, x, kc, vc, ks, vs, shared, x.context_lens)
    b = _decode_codes(fmt, x, kq, vq, ks, vs, x.block_table, x.context_lens)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2), (16, 2), (32, 2), (24, 2)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_head_dim_64_and_wide_groups(fmt, hq, hkv, dtype):
    # head_dim 64 pools (64-byte code rows) and GQA groups of 1 to 16 query
    # heads per KV head (24: one full and one partly filled 16-head slice).
    lengths = [0, 1, 15, 17, 33, 200, 333]
    for d, bs in ((64, 16), (64, 128), (128, 32)):
        c = cfg(hq=hq, hkv=hkv, d=d, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 8,
                dtype=dtype, lengths=lengths)
        x = W.make_inputs(c, seed=700 + hq + hkv + d + bs)
        for part in (0, 64):
            check_decode(fmt, x, part, f"d{d} bs{bs} g{hq // hkv} {dtype} P{part}")


@pytest.mark.parametrize("fmt", FORMATS)
def test_llama7b_shape_at_head_dim_64(fmt):
    # llama7b-decode's batch, lengths and pool with 64-wide heads.
    x = W.make_inputs("llama7b-decode", head_dim=64)
    check_decode(fmt, x, 0, "llama7b d64")


@pytest.mark.parametrize("fmt", FORMATS)
def test_bf16_queries_outside_fp16_range(fmt):
    # bf16 queries keep their own range: heads 0-3 beyond fp16's largest
    # finite value (65504), heads 4-7 below its smallest normal (2^-14).
    # One-byte codes widen exactly to bf16, so the query is never rounded.
    require_gpu()
    x = W.make_inputs(cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16",
                          lengths=[40, 90, 17, 128]), seed=77)
    q = x.q.float()
    q[:, :4] *= 3.0e5
    q[:, 4:] *= 1.0e-7
    x.q = q.to(torch.bfloat16)
    assert (x.q[:, :4].float().abs().max() > 65504) and (x.q[:, 4:].float().abs().max() < 2**-14)
    check_decode(fmt, x, 0, "bf16 query range")
    check_decode(fmt, x, 64, "bf16 query range P64")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("d,hq,hkv", [(64, 8, 2), (128, 32, 2)])
def test_decode_write_step_shapes(fmt, d, hq, hkv):
    """The one-call 8-bit step at head_dim 64 and with 16 query heads per KV
    head: pools equal to the oracle's write, output within tolerance of the
    oracle's decode over those codes."""
    require_gpu()
    c = cfg(hq=hq, hkv=hkv, d=d, bs=16, nb=200, dtype="bf16", lengths=[1, 40, 300, 17, 1000],
            write_new_token=True)
    x = W.make_inputs(c, seed=88 + d + hq)
    kc, vc, ks, vs = pools8(x, fmt)  # the codes after this step's write
    slots = x.slot_mapping.numpy()
    k0, v0 = kc.copy(), vc.copy()
    k0.reshape(-1, hkv, d)[slots] = 0  # before the write
    v0.reshape(-1, hkv, d)[slots] = 0
    for part in (0, 64):
        kd, vd, err = torch.from_numpy(k0.copy()).cuda(), torch.from_numpy(v0.copy()).cuda(), \
            new_err()
        q = x.q.cuda()
        out = torch.full_like(q, float("nan"))
        GPU_STEP[fmt](out, q, x.k_new.cuda(), x.v_new.cuda(), kd, vd, x.slot_mapping.cuda(),
                      x.block_table.cuda(), x.context_lens.cuda(), ks.cuda(), vs.cuda(),
                      scale=x.scale, max_context_len=x.max_context_len, partition_size=part,
                      d_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert np.array_equal(kd.cpu().numpy(), kc) and np.array_equal(vd.cpu().numpy(), vc)
        assert_close(out, oracle_decode8(fmt, x, kc, vc, ks, vs), x.dtype,
                     what=f"{fmt} step d{d} g{hq // hkv} P{part}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_quantiser_every_input_pattern(fmt, dtype):
    """The write's quantiser over every 16-bit input pattern (NaN, infinities,
    signed zeros and subnormals included) and scales from 2^-130 to 2^20,
    odd mantissas among them: codes bit-identical to the oracle's, whose
    quotient is the IEEE fp32 division x / scale."""
    require_gpu()
    pats = np.arange(65536, dtype=np.uint16)
    t16 = TORCH16[oracle.F16 if dtype == "f16" else oracle.BF16]
    x = torch.from_numpy(pats.view(np.int16)).view(t16)
    hkv, d = 4, 128
    rows = x.reshape(-1, hkv, d)                      # 128 tokens of 4 heads
    n = rows.shape[0]
    scales = [2.0 ** -130, 1.0e-38, 3.0e-12, 0.0123, 0.0078125, 1.0 / 3.0, 1.7, 1024.5,
              2.0 ** 20]
    for s in scales:
        sc = torch.full((hkv,), s, dtype=torch.float32)
        kd = torch.zeros((n, 1, hkv, d), dtype=torch.int8 if fmt == "int8" else torch.uint8,
                         device="cuda")
        vd = torch.zeros_like(kd)
        slots = torch.arange(n, dtype=torch.int64, device="cuda")
        GPU_WRITE[fmt](rows.cuda(), rows.flip(0).contiguous().cuda(), kd, vd, slots, sc.cuda(),
                       sc.cuda())
        torch.cuda.synchronize()
        want = QUANTIZE[fmt](x, float(np.float32(s))).reshape(n, 1, hkv, d)
        got = kd.cpu().numpy()
        bad = np.flatnonzero(got.reshape(-1) != want.reshape(-1))
        assert bad.size == 0, (f"{fmt} {dtype} scale {s}: {bad.size} codes differ, first input "
                               f"pattern {int(pats[bad[0]]):#06x}")
        assert np.array_equal(vd.cpu().numpy(), want[::-1])
