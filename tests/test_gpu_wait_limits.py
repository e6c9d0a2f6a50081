"""The kernels' bounded waits run out without a fault, and the launches after
them are unaffected.

Every pipeline wait in the decode and prefill kernels is bounded; when one
runs out the kernel sets PA_DEVERR_TIMEOUT, waits for its own copies in
flight, frees its tensor memory (prefill), still counts itself into the
prefill's work-counter slot, and returns.  pa_debug_set_wait_limit_ns
shortens the bound so these tests can make waits run out on purpose (no
fault, no hang: the waits for copies in flight keep their 2 s bound).  The
launches that follow -- enough prefill launches to reuse every one of the
256 work-counter slots, including the one the timed-out launch used -- must
give the same bits as before."""
import pytest
import torch

from gpu_util import (W, assert_close, cfg, gpu, gpu_decode, gpu_prefill, gpu_write, new_err,
                      oracle_pools_after_write, oracle_prefill, pa, require_gpu)

pytestmark = gpu

SLOTS = 256  # prefill work-counter slots, taken round robin


def test_waits_run_out_and_later_launches_are_unaffected():
    require_gpu()
    xp_host = W.make_inputs(cfg(kind="prefill", hq=8, hkv=2, d=128, bs=32, nb=200,
                                dtype="bf16", lengths=[700, 300, 1000, 64]), seed=81)
    xp = xp_host.to("cuda")
    gpu_write(xp)
    xd = W.make_inputs("llama7b-decode", device="cuda")
    gpu_write(xd)
    ref_p = gpu_prefill(xp)
    ref_d = gpu_decode(xd)
    torch.cuda.synchronize()
    try:
        pa.pa_debug_set_wait_limit_ns(1)  # a wait not met at its first try runs out
        err_p, err_d = new_err(), new_err()
        gpu_prefill(xp, err=err_p)
        gpu_decode(xd, err=err_d)
        torch.cuda.synchronize()
    finally:
        pa.pa_debug_set_wait_limit_ns(0)
    assert int(err_p.item()) & pa.DEVERR_TIMEOUT
    assert int(err_d.item()) & pa.DEVERR_TIMEOUT
    # the next launches, on the same stream: every work-counter slot again
    for i in range(SLOTS + 8):
        err = new_err()
        out = gpu_prefill(xp, err=err)
        if i % 32 == 0 or i >= SLOTS:
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            assert torch.equal(out.view(torch.int16), ref_p.view(torch.int16)), f"launch {i}"
    err = new_err()
    out_d = gpu_decode(xd, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out_d.view(torch.int16), ref_d.view(torch.int16))
    kp, vp = oracle_pools_after_write(xp_host)
    assert_close(out, oracle_prefill(xp_host, kp, vp), xp_host.dtype, what="after timeouts")


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_default_bound_restored(kind):
    # 0 restores the 2 s default: ordinary launches report no timeout.
    require_gpu()
    pa.pa_debug_set_wait_limit_ns(0)
    err = new_err()
    if kind == "decode":
        gpu_decode(W.make_inputs("continuous-batching", device="cuda"), err=err)
    else:
        x = W.make_inputs("packed-prefill", device="cuda")
        gpu_write(x)
        gpu_prefill(x, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
