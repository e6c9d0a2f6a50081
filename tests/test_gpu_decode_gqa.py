"""pa_decode for every GQA ratio Hq % Hkv == 0 on the GPU, against the fp64
oracle element by element.

The pages fix only num_key_value_heads as a parameter (cannbot-skills page
§2, mode 2 FA parameters), with no bound on the group G = Hq / Hkv; query
head h reads KV head h / G.  The kernel serves up to 16 query heads of a KV
head from one K/V read (two 8-head column groups of the score tile) and
wider groups in 16-head slices; these cases cover one and two column groups,
partly filled groups (G = 10, 12, 24) and several slices (G = 24, 32, 64)."""
import numpy as np
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, gpu_decode, gpu_write, new_err,
                      oracle_decode, oracle_pools_after_write, require_gpu, u16)

pytestmark = gpu


def _run(x_host, partition_size, what, want=None):
    require_gpu()
    if want is None:
        kp, vp = oracle_pools_after_write(x_host)
        want = oracle_decode(x_host, kp, vp)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    out = gpu_decode(x, partition_size=partition_size, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"{what}: device error bits {int(err.item())}"
    return out, assert_close(out, want, x.dtype, what=what)


@pytest.mark.parametrize("hq,hkv", [(40, 4), (24, 2), (64, 4), (48, 2), (128, 4), (64, 1)])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [16, 128])
def test_group_grid(hq, hkv, d, bs):
    lengths = [0, 1, bs - 1, bs + 1, 300, 1000, 77]
    c = cfg(hq=hq, hkv=hkv, d=d, bs=bs, nb=sum(-(-n // bs) for n in lengths) + 4,
            dtype="bf16" if (hq + d + bs) % 2 else "f16", lengths=lengths)
    x = W.make_inputs(c, seed=500 + hq + hkv + d + bs)
    for part in (0, 64, 512):
        _run(x, part, f"G{hq // hkv} hkv{hkv} d{d} bs{bs} P{part}")


@pytest.mark.parametrize("hq,hkv", [(64, 4), (128, 4)])
def test_long_context_wide_groups_full_outputs(hq, hkv):
    # The long-context workload's shape and lengths (4 sequences of 32K-128K
    # tokens, bs 128, 512-token partitions) with 16 and 32 query heads per KV
    # head; every output element against the oracle.
    require_gpu()
    x = W.make_inputs("long-context-decode", num_q_heads=hq, num_kv_heads=hkv)
    kp, vp = oracle_pools_after_write(x)
    want = oracle_decode(x, kp, vp)
    for part in (x.partition_size, 0):
        _run(x, part, f"long-context G{hq // hkv} P{part}", want)


def test_continuous_batching_group_16():
    # The continuous-batching workload (32 sequences, log-uniform lengths,
    # shuffled free list) with 128 query heads over 8 KV heads.
    x = W.make_inputs("continuous-batching", num_q_heads=128)
    _run(x, 0, "continuous-batching G16")


def test_wide_group_equals_narrow_groups_bitwise():
    # A KV head's query heads are independent: the 16 heads of a G = 16 call
    # equal, bit for bit, the same heads split over two G = 8 calls that
    # read the same KV head (each call serves 8 of the 16 query heads).
    require_gpu()
    x = W.make_inputs(cfg(hq=32, hkv=2, d=128, bs=16, nb=200, dtype="bf16",
                          lengths=[700, 1500, 33, 1]), seed=61)
    wide = gpu_decode(x.to("cuda"), partition_size=256)
    q = x.q.view(x.num_seqs, 2, 16, 128)  # [S, KV head, 16 heads, D]
    outs = []
    for half in range(2):
        y = x.to("cpu")
        y.q = q[:, :, 8 * half:8 * half + 8].reshape(x.num_seqs, 16, 128).contiguous()
        y.num_q_heads = 16
        outs.append(gpu_decode(y.to("cuda"), partition_size=256).cpu()
                    .view(x.num_seqs, 2, 8, 128))
    torch.cuda.synchronize()
    narrow = torch.cat(outs, dim=2).reshape(x.num_seqs, 32, 128)
    assert np.array_equal(u16(wide.cpu()), u16(narrow))
