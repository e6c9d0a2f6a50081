"""pa_reshape_and_cache on the GPU against the oracle's write: bit-exact over
the whole pool (untouched rows keep their NaN sentinel)."""
import numpy as np
import pytest
import torch

from gpu_util import (W, cfg, gpu, gpu_write, new_err, oracle_pools_after_write, pa,
                      require_gpu, u16)

pytestmark = gpu


def _check_write(x_host):
    require_gpu()
    want_k, want_v = oracle_pools_after_write(x_host)
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(u16(x.k_pool), want_k)
    assert np.array_equal(u16(x.v_pool), want_v)


@pytest.mark.parametrize("name", ["llama7b-decode", "packed-prefill"])
def test_named_config_write_pattern(name):
    _check_write(W.make_inputs(name))


@pytest.mark.parametrize("name", ["tiny-decode", "continuous-batching"])
def test_decode_configs_with_new_token_write(name):
    _check_write(W.make_inputs(name, write_new_token=True))


@pytest.mark.parametrize("hkv,d,bs,dtype", [(2, 64, 16, "f16"), (8, 128, 32, "f16"),
                                            (1, 64, 8, "bf16"), (3, 128, 128, "bf16"),
                                            (32, 128, 16, "bf16")])
def test_shapes_and_dtypes(hkv, d, bs, dtype):
    c = cfg(kind="prefill", hq=hkv, hkv=hkv, d=d, bs=bs, nb=64, dtype=dtype,
            lengths=[1, bs - 1, bs, bs + 1, 3 * bs + 5])
    _check_write(W.make_inputs(c, seed=5))


def test_negative_slots_skipped_and_last_slot_written():
    require_gpu()
    x = W.make_inputs(cfg(kind="prefill", hq=2, hkv=2, d=64, bs=16, nb=8,
                          lengths=[20, 30], dtype="f16"), seed=9)
    slots = x.slot_mapping.clone()
    slots[::3] = -1
    slots[1] = x.num_blocks * x.block_size - 1  # the pool's very last row
    x.slot_mapping = slots
    _check_write(x)


def test_bad_slot_flagged_and_skipped():
    require_gpu()
    x = W.make_inputs(cfg(kind="prefill", hq=2, hkv=2, d=64, bs=16, nb=8,
                          lengths=[10], dtype="f16"), seed=11)
    slots = x.slot_mapping.clone()
    slots[4] = x.num_blocks * x.block_size  # one past the end
    x_host = x
    x_host.slot_mapping = slots
    kp, vp = u16(x_host.k_pool).copy(), u16(x_host.v_pool).copy()
    import oracle
    assert oracle.write(kp, vp, x_host.k_new, x_host.v_new, slots, 16) == oracle.ERR_SLOT
    x = x_host.to("cuda")
    err = new_err()
    gpu_write(x, err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.DEVERR_SLOT
    assert np.array_equal(u16(x.k_pool), kp) and np.array_equal(u16(x.v_pool), vp)


def test_interleaved_qkv_rows():
    # K and V as views into a [N, 3, H, D] buffer (row stride 3*H*D).
    require_gpu()
    x = W.make_inputs(cfg(kind="prefill", hq=4, hkv=4, d=128, bs=32, nb=16,
                          lengths=[40, 70], dtype="bf16"), seed=13)
    n = x.k_new.shape[0]
    qkv = torch.empty(n, 3, 4, 128, dtype=x.dtype)
    qkv[:, 1] = x.k_new
    qkv[:, 2] = x.v_new
    want_k, want_v = oracle_pools_after_write(x)
    xd = x.to("cuda")
    qkv = qkv.cuda()
    pa.pa_reshape_and_cache(qkv[:, 1], qkv[:, 2], xd.k_pool, xd.v_pool, xd.slot_mapping)
    torch.cuda.synchronize()
    assert np.array_equal(u16(xd.k_pool), want_k) and np.array_equal(u16(xd.v_pool), want_v)
