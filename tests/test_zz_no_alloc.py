"""pa_decode_static_ws: decode without a caller-supplied workspace.

The entry point exists for callers that cannot allocate device memory (code
that must not call cudaMalloc, a fixed memory budget, a host framework that
owns every allocation, a plain C caller).  It must give the same results as
pa_decode with an allocated workspace.  These tests call both through the C
ABI on the same inputs, twice in a row with different inputs (the shared
device array keeps the previous call's contents), and once where the
automatic plan has to be lengthened to fit the array.  Each output is also
checked against the fp64 oracle of the same step (its own write, then its
decode) within the dtype's bound.

This file is collected last on purpose: it also passes when run alone."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_34_gb300 as pa
from gpu_util import assert_close, oracle_decode, oracle_pools_after_write
from paged_kv_cache_34_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
STATIC_BYTES = 16 << 20  # PA_STATIC_WORKSPACE_BYTES


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = pa.library()
    c = ctypes
    V, I32, I64, F = c.c_void_p, c.c_int32, c.c_int64, c.c_float
    lib.pa_decode_static_ws.argtypes = [V, I64, V, I64, V, V, V, I64, I32, V, I32, I32, I32,
                                        I32, I32, I64, F, I32, I32, c.c_int, V, V]
    lib.pa_decode_static_ws.restype = c.c_int
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def static_decode(lib, x, out, partition_size, err):
    s, hq, d = x.q.shape
    nb, bs, hkv, _ = x.k_pool.shape
    return lib.pa_decode_static_ws(
        _ptr(out), out.stride(0), _ptr(x.q), x.q.stride(0), _ptr(x.k_pool), _ptr(x.v_pool),
        _ptr(x.block_table), x.block_table.stride(0), x.block_table.shape[1],
        _ptr(x.context_lens), s, hq, hkv, d, bs, nb, x.scale, x.max_context_len, partition_size,
        1 if x.dtype == torch.bfloat16 else 0, _ptr(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def inputs(name, with_oracle=True, **kw):
    """Seeded inputs with the step's new tokens already in the cache (decode
    reads the cache after the write, so context_lens count them), and the
    oracle's output for them (from the host copies: the oracle's own write,
    then its decode)."""
    x_host = W.make_inputs(name, **kw)
    x = x_host.to("cuda")
    if x.slot_mapping.numel():
        pa.pa_reshape_and_cache(x.k_new, x.v_new, x.k_pool, x.v_pool, x.slot_mapping)
    if with_oracle:
        kp, vp = oracle_pools_after_write(x_host)
        x.want = oracle_decode(x_host, kp, vp)
    return x


def allocated_decode(x, partition_size):
    out = torch.empty_like(x.q)
    pa.pa_decode(out, x.q, x.k_pool, x.v_pool, x.block_table, x.context_lens, scale=x.scale,
                 max_context_len=x.max_context_len, partition_size=partition_size)
    return out


def check(lib, x, partition_size=0):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(x.q, float("nan"))
    assert static_decode(lib, x, out, partition_size, err) == 0
    want = allocated_decode(x, partition_size)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(out).all()
    diff = (out.double() - want.double()).abs().max().item()
    assert diff <= TOL[x.dtype], f"max-abs difference {diff}"
    assert_close(out, x.want, x.dtype, what="static workspace vs oracle")
    return out


def test_two_calls_in_a_row_match_pa_decode():
    lib = _lib()
    # 1: many partitions per sequence (the array holds partial results)
    a = inputs("llama7b-decode")
    P, need = pa.pa_decode_plan(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim,
                                a.max_context_len, 64)
    assert 0 < need <= STATIC_BYTES
    out_a = check(lib, a, partition_size=64)
    # 2: different shapes and dtype right after, reusing the same array
    b = inputs("continuous-batching")
    check(lib, b, partition_size=128)
    # 1 again: identical to the first call (no state carried over)
    again = torch.empty_like(a.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert static_decode(lib, a, again, 64, err) == 0
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), out_a.view(torch.int16))


def test_automatic_plan_falls_back_to_fixed_partitions_that_fit():
    lib = _lib()
    # 512 short sequences with 8 query heads per KV head: the automatic
    # (balanced) plan keeps one partial state per query head per piece, more
    # than the array holds, so the call switches to fixed partitions grown
    # until they fit.
    lengths = [64 + (37 * i) % 400 for i in range(512)]
    x = inputs("long-context-decode", num_seqs=512, lengths=lengths)
    _, need = pa.pa_decode_plan(x.num_seqs, x.num_q_heads, x.num_kv_heads, x.head_dim,
                                x.max_context_len, 0)
    assert need > STATIC_BYTES  # the automatic plan would not fit
    check(lib, x, partition_size=0)
    # an explicit partition size that does not fit is refused, not run
    y = inputs("long-context-decode", with_oracle=False,
               lengths=[131072, 120000, 90000, 131000])
    _, need64 = pa.pa_decode_plan(y.num_seqs, y.num_q_heads, y.num_kv_heads, y.head_dim,
                                  y.max_context_len, 64)
    assert need64 > STATIC_BYTES
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(y.q)
    assert static_decode(lib, y, out, 64, err) == 5  # PA_ERR_WORKSPACE
