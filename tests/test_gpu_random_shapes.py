"""Seeded random shapes against the fp64 oracle, every output row.

Each case draws a small batch -- query/KV head counts (GQA groups from 1 to
16, powers of two and not), head_dim, block size, dtype, ragged context
lengths including 0 and block/tile edges, and the split plan -- and checks
the decode (16-bit pools, the one-call step, INT8 and FP8 pools) or the
prefill (whole sequences and chunks, causal and not) against the oracle
within the dtype's tolerance.  The draws are fixed by the seed, so a failure
names a reproducible case."""
import numpy as np
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, gpu_decode, gpu_prefill, gpu_write, new_err,
                      oracle_decode, oracle_pools_after_write, oracle_prefill, pa, require_gpu,
                      u16)
from test_gpu_kv8 import check_decode as check_decode8

pytestmark = gpu

GROUPS = [(4, 4), (8, 4), (8, 2), (12, 4), (16, 2), (24, 2), (32, 2), (40, 8), (64, 4),
          (16, 16)]


def _draw(seed, kind):
    r = np.random.default_rng(seed)
    hq, hkv = GROUPS[int(r.integers(len(GROUPS)))]
    d = int(r.choice([64, 128]))
    bs = int(r.choice([16, 32, 64, 128] if kind == "prefill" else [8, 16, 32, 64, 128]))
    dtype = str(r.choice(["f16", "bf16"]))
    n = int(r.integers(1, 7))
    top = 700 if kind == "prefill" else 1500
    lengths = [int(v) for v in r.integers(0 if kind == "decode" else 1, top, size=n)]
    # a few lengths on block and tile edges
    for i in range(n):
        if r.random() < 0.3:
            lengths[i] = int(r.choice([1, bs - 1, bs, bs + 1, 127, 128, 129, 256]))
            lengths[i] = max(lengths[i], 0 if kind == "decode" else 1)
    nb = sum(-(-L // bs) for L in lengths) + int(r.integers(1, 8))
    return r, dict(hq=hq, hkv=hkv, d=d, bs=bs, nb=nb, dtype=dtype, lengths=lengths)


def _what(c, extra=""):
    return (f"{c['hq']}/{c['hkv']} d{c['d']} bs{c['bs']} {c['dtype']} "
            f"L={c['lengths']} {extra}")


@pytest.mark.parametrize("seed", range(24))
def test_random_decode(seed):
    require_gpu()
    r, c = _draw(1000 + seed, "decode")
    part = int(r.choice([0, 0, 64, 256]))
    x_host = W.make_inputs(cfg(**c, write_new_token=True), seed=2000 + seed)
    kp, vp = oracle_pools_after_write(x_host)
    want = oracle_decode(x_host, kp, vp)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    out = gpu_decode(x, partition_size=part, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert_close(out, want, x.dtype, what=_what(c, f"P{part}"))


@pytest.mark.parametrize("seed", range(12))
def test_random_decode_step(seed):
    # the one-call step: this step's rows written, then the decode that reads
    # them; pools bit-exact, output against the oracle
    require_gpu()
    r, c = _draw(3000 + seed, "decode")
    part = int(r.choice([0, 0, 64]))
    x_host = W.make_inputs(cfg(**c, write_new_token=True), seed=4000 + seed)
    kp, vp = oracle_pools_after_write(x_host)
    want = oracle_decode(x_host, kp, vp)
    x = x_host.to("cuda")
    err = new_err()
    out = torch.full_like(x.q, float("nan"))
    pa.pa_decode_write(out, x.q, x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                       x.block_table, x.context_lens, scale=x.scale,
                       max_context_len=x.max_context_len, partition_size=part, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert np.array_equal(u16(x.k_pool), kp) and np.array_equal(u16(x.v_pool), vp)
    assert_close(out, want, x.dtype, what=_what(c, f"step P{part}"))


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("seed", range(8))
def test_random_decode_one_byte_pools(fmt, seed):
    r, c = _draw(5000 + seed, "decode")
    part = int(r.choice([0, 64]))
    x = W.make_inputs(cfg(**c, write_new_token=True), seed=6000 + seed)
    check_decode8(fmt, x, part, _what(c, f"P{part}"))


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill(seed):
    require_gpu()
    r, c = _draw(7000 + seed, "prefill")
    causal = bool(r.random() < 0.75)
    chunked = bool(r.random() < 0.5)
    qlens = [int(r.integers(1, L + 1)) if chunked else L for L in c["lengths"]]
    x_host = W.make_inputs(cfg(kind="prefill", causal=causal, **c), seed=8000 + seed,
                           q_lens=qlens, new_lens=qlens)
    kp, vp = oracle_pools_after_write(x_host)
    want = oracle_prefill(x_host, kp, vp)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    out = gpu_prefill(x, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    assert_close(out, want, x.dtype, what=_what(c, f"q={qlens} causal={causal}"))
