"""pa_decode_write on the GPU: one decode step (the new tokens' cache write,
then the decode that reads them) as one call.

It must equal pa_reshape_and_cache followed by pa_decode bit for bit (same
kernels, same split; only the overlap of the two differs) -- pools and
output -- and match the fp64 oracle of write-then-decode ([SKILL] §3.6:
write this step's K/V, then attend with context_lens that count it)."""
import numpy as np
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, new_err, oracle_decode,
                      oracle_pools_after_write, pa, require_gpu, u16)

pytestmark = gpu


def fused(x, partition_size, err=None):
    out = torch.full_like(x.q, float("nan"))
    pa.pa_decode_write(out, x.q, x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                       x.block_table, x.context_lens, scale=x.scale,
                       max_context_len=x.max_context_len, partition_size=partition_size,
                       d_error=err)
    return out


def separate(x, partition_size, err=None):
    out = torch.full_like(x.q, float("nan"))
    if x.slot_mapping.numel():
        pa.pa_reshape_and_cache(x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                                d_error=err)
    pa.pa_decode(out, x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens, scale=x.scale,
                 max_context_len=x.max_context_len, partition_size=partition_size, d_error=err)
    return out


def check(x_host, partition_size, what):
    require_gpu()
    a, b = x_host.to("cuda"), x_host.to("cuda")
    ea, eb = new_err(), new_err()
    got = fused(a, partition_size, ea)
    want_gpu = separate(b, partition_size, eb)
    torch.cuda.synchronize()
    assert int(ea.item()) == 0 and int(eb.item()) == 0
    # bit-identical to the two calls, pools included
    assert np.array_equal(u16(got), u16(want_gpu)), what
    assert np.array_equal(u16(a.k_pool), u16(b.k_pool))
    assert np.array_equal(u16(a.v_pool), u16(b.v_pool))
    # and the oracle of write-then-decode (the pools bit for bit)
    kp, vp = oracle_pools_after_write(x_host)
    assert np.array_equal(u16(a.k_pool), kp) and np.array_equal(u16(a.v_pool), vp)
    assert_close(got, oracle_decode(x_host, kp, vp), x_host.dtype, what=what)


@pytest.mark.parametrize("partition_size", [0, 64, 256])
def test_llama7b_step_matches_separate_calls_and_oracle(partition_size):
    check(W.make_inputs("llama7b-decode"), partition_size, f"llama7b P{partition_size}")


@pytest.mark.parametrize("bs,hq,hkv,dtype,d", [(16, 8, 2, "f16", 128), (32, 32, 8, "bf16", 128),
                                               (128, 64, 8, "bf16", 128), (8, 4, 4, "f16", 128),
                                               (16, 64, 4, "bf16", 128), (32, 64, 2, "f16", 64),
                                               (16, 8, 1, "bf16", 64)])
def test_gqa_and_block_sizes(bs, hq, hkv, dtype, d):
    lengths = [1, bs - 1, bs, bs + 1, 63, 200, 333]
    c = cfg(hq=hq, hkv=hkv, d=d, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 8,
            dtype=dtype, lengths=lengths, write_new_token=True)
    x = W.make_inputs(c, seed=7 + bs + hq)
    for part in (0, 64):
        check(x, part, f"bs{bs} g{hq // hkv} d{d} {dtype} P{part}")


def test_step_rows_not_the_newest():
    # One new token per sequence, but slot_mapping does not send every token
    # to its own sequence's newest position: sequence 1 writes nothing this
    # step (slot -1, and its context excludes the token), and tokens 2 and 3
    # are sent to each other's newest slot.  The step must still equal the
    # write followed by the decode (the decode reads those newest rows from
    # the pool once the write has finished).
    c = cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16", lengths=[40, 90, 17, 33, 64],
            write_new_token=True)
    x = W.make_inputs(c, seed=13)
    sm = x.slot_mapping.clone()
    sm[1] = -1
    sm[2], sm[3] = x.slot_mapping[3].item(), x.slot_mapping[2].item()
    x.slot_mapping = sm
    x.context_lens = x.context_lens.clone()
    x.context_lens[1] -= 1
    for part in (0, 64):
        check(x, part, f"crossed slots P{part}")


def test_padding_slots_and_empty_sequences():
    # a sequence with no new token this step (slot -1) and an empty sequence
    c = cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16", lengths=[0, 40, 90, 17],
            write_new_token=True)
    x = W.make_inputs(c, seed=11)
    # new tokens are listed for the non-empty sequences 1, 2, 3 in order
    sm = x.slot_mapping.clone()
    sm[0] = -1  # sequence 1's new row is not written: its last pool row stays NaN
    x.slot_mapping = sm
    x.context_lens = x.context_lens.clone()
    x.context_lens[1] -= 1  # ... so it attends one key fewer
    check(x, 0, "padding slot")


def test_no_new_tokens_is_plain_decode():
    require_gpu()
    x = W.make_inputs("continuous-batching", device="cuda")
    empty = torch.zeros(0, dtype=torch.int64, device="cuda")
    k0 = x.k_new[:0]
    out = torch.empty_like(x.q)
    pa.pa_decode_write(out, x.q, k0, k0, x.k_pool, x.v_pool, empty, x.block_table,
                       x.context_lens, scale=x.scale, max_context_len=x.max_context_len)
    ref = torch.empty_like(x.q)
    pa.pa_decode(ref, x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens, scale=x.scale,
                 max_context_len=x.max_context_len)
    torch.cuda.synchronize()
    assert np.array_equal(u16(out), u16(ref))


def test_device_errors_flagged():
    # a slot past the pool: PA_DEVERR_SLOT from the write half, the decode runs
    require_gpu()
    c = cfg(hq=8, hkv=2, d=128, bs=16, nb=64, dtype="bf16", lengths=[30, 50],
            write_new_token=True)
    x = W.make_inputs(c, seed=5).to("cuda")
    sm = x.slot_mapping.clone()
    sm[0] = 64 * 16 + 3
    x.slot_mapping = sm
    err = new_err()
    out = fused(x, 0, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SLOT
    assert torch.isfinite(out[1]).all()
