"""Helpers shared by the GPU parity tests: run one op of the CUDA library on
seeded inputs, and compare with the fp64 oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_34_gb300 as pa
from paged_kv_cache_34_gb300 import workloads as W

# Max-abs error bounds against the fp64 oracle.
TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}

gpu = pytest.mark.gpu


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def u16(t):
    return oracle._u16(t)


def new_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gpu_write(x, err=None):
    """Apply the step's cache write on the device pools (in place)."""
    if x.slot_mapping.numel():
        pa.pa_reshape_and_cache(x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping,
                                d_error=err)


def oracle_pools_after_write(x_host):
    """Host uint16 pools with the step's write applied by the oracle."""
    kp, vp = u16(x_host.k_pool).copy(), u16(x_host.v_pool).copy()
    if x_host.slot_mapping.numel():
        st = oracle.write(kp, vp, x_host.k_new, x_host.v_new, x_host.slot_mapping,
                          x_host.block_size)
        assert st == oracle.OK
    return kp, vp


def gpu_decode(x, partition_size=None, err=None, max_context_len=None, out=None):
    if out is None:
        out = torch.empty_like(x.q)
    pa.pa_decode(out, x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens, scale=x.scale,
                 max_context_len=(x.max_context_len if max_context_len is None
                                  else max_context_len),
                 partition_size=(x.partition_size if partition_size is None
                                 else partition_size), d_error=err)
    return out


def gpu_prefill(x, err=None, out=None):
    if out is None:
        out = torch.empty_like(x.q)
    pa.pa_prefill_varlen(out, x.q, x.k_pool, x.v_pool, x.block_table, x.cu_seqlens_q,
                         x.context_lens, scale=x.scale, max_seqlen_q=x.max_seqlen_q,
                         max_context_len=x.max_context_len, causal=x.causal, d_error=err)
    return out


def oracle_decode(x_host, kp, vp):
    return oracle.decode(x_host.q, kp, vp, x_host.block_table, x_host.context_lens,
                         x_host.num_kv_heads, x_host.block_size, x_host.scale,
                         dtype=oracle.dtype_code(x_host.dtype))


def oracle_prefill(x_host, kp, vp, rows=None):
    return oracle.prefill(x_host.q, kp, vp, x_host.block_table, x_host.cu_seqlens_q,
                          x_host.context_lens, x_host.num_kv_heads, x_host.block_size,
                          x_host.scale, causal=x_host.causal, rows=rows,
                          dtype=oracle.dtype_code(x_host.dtype))


# significand bits (with the implicit one) of the output types
SIG_BITS = {torch.float16: 11, torch.bfloat16: 8}


def bound(want, dtype):
    """Per-element max-abs bound: the stated one (TOL), except where half an
    ulp of the output type at the exact value -- the error of rounding the
    exact result itself -- leaves no room under it (bf16 from |o| >= 4, fp16
    from |o| >= 4): there, that half ulp plus a fifth of the stated bound for
    the kernel's own arithmetic."""
    a = np.abs(want)
    e = np.floor(np.log2(np.maximum(a, np.finfo(np.float64).tiny)))
    half_ulp = np.exp2(e - SIG_BITS[dtype])
    return np.maximum(TOL[dtype], half_ulp + TOL[dtype] / 5)


def assert_close(got, want, dtype, rows=None, what=""):
    g = got.detach().double().cpu().numpy()
    if rows is not None:
        g, want = g[rows], want[rows]
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - want)
    err = d.max(initial=0.0)
    over = d > bound(want, dtype)
    if over.any():
        i = np.unravel_index(np.argmax(np.where(over, d, -1.0)), d.shape)
        raise AssertionError(f"{what}: max-abs error {d[i]:.3g} at {tuple(int(k) for k in i)} "
                             f"(expected {want[i]:.6g}) > bound {bound(want[i], dtype):.3g}")
    return err


def cfg(kind="decode", hq=8, hkv=2, d=128, bs=16, nb=256, dtype="bf16", lengths=None,
        placement="permutation", seqs=None, **extra):
    c = dict(kind=kind, num_seqs=len(lengths) if seqs is None else seqs,
             lengths=("list", list(lengths), None), num_q_heads=hq, num_kv_heads=hkv,
             head_dim=d, block_size=bs, num_blocks=nb, placement=placement, dtype=dtype,
             name="case")
    c.update(extra)
    return c


__all__ = ["TOL", "gpu", "require_gpu", "new_err", "gpu_write", "oracle_pools_after_write",
           "gpu_decode", "gpu_prefill", "oracle_decode", "oracle_prefill", "assert_close",
           "cfg", "W", "pa", "u16"]
