"""Attention over a paged KV cache on NVIDIA GB300 (sm_103a).

Python binding of ``libpa.so``, the C-ABI CUDA library declared in
``include/pa.h``.  Each function here only marshals torch tensors into the
C call (device pointers, sizes, strides, the current CUDA stream) and turns a
non-OK status into an exception; every step of the computation runs in the
library's kernels.  There is no CPU fallback: without the built library the
first call raises.

    pa_reshape_and_cache  new K/V rows -> pool rows given by slot_mapping
    pa_decode             one query per sequence, split-KV + LSE combine
    pa_prefill_varlen     causal attention for cu_seqlens-packed queries
    pa_reshape_and_cache_int8, pa_decode_int8, pa_decode_write_int8 (and _fp8)
                          the write, decode and step over INT8 (FP8 E4M3) pools
    pa_copy_blocks        copy whole blocks of both pools (copy-on-write)

Build the library with ``python -m paged_kv_cache_34_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["pa_reshape_and_cache", "pa_decode", "pa_decode_plan", "pa_decode_write",
           "pa_prefill_varlen", "pa_reshape_and_cache_int8", "pa_decode_int8",
           "pa_decode_write_int8", "pa_reshape_and_cache_fp8", "pa_decode_fp8",
           "pa_decode_write_fp8", "pa_copy_blocks", "PaError",
           "library", "DEVERR_SLOT", "DEVERR_BLOCK_ID", "DEVERR_CU_SEQLENS",
           "DEVERR_CONTEXT", "DEVERR_TIMEOUT", "DEVERR_SCALE", "LIB_PATH"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

# Device error bits (include/pa.h PA_DEVERR_*).
DEVERR_SLOT, DEVERR_BLOCK_ID, DEVERR_CU_SEQLENS, DEVERR_CONTEXT, DEVERR_TIMEOUT = 1, 2, 4, 8, 16
DEVERR_SCALE = 32

_STATUS = {0: "PA_OK", 1: "PA_ERR_NULL", 2: "PA_ERR_SHAPE", 3: "PA_ERR_UNSUPPORTED",
           4: "PA_ERR_ALIGN", 5: "PA_ERR_WORKSPACE", 6: "PA_ERR_CUDA"}
_DTYPE = {torch.float16: 0, torch.bfloat16: 1}


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lock = threading.Lock()
_lib = None


def library(path: str | None = None):
    """The loaded libpa.so (ctypes), with argument types declared."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is not built; run `python -m paged_kv_cache_34_gb300.build` "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(p)
        c = ctypes
        V, I32, I64, F, SZ = c.c_void_p, c.c_int32, c.c_int64, c.c_float, c.c_size_t
        lib.pa_abi_version.argtypes, lib.pa_abi_version.restype = [], I32
        lib.pa_status_string.argtypes, lib.pa_status_string.restype = [c.c_int], c.c_char_p
        lib.pa_last_cuda_error.argtypes, lib.pa_last_cuda_error.restype = [], I32
        lib.pa_debug_set_wait_limit_ns.argtypes = [c.c_uint64]
        lib.pa_debug_set_wait_limit_ns.restype = None
        lib.pa_reshape_and_cache.argtypes = [V, V, I64, V, V, V, I32, I32, I32, I32, I64,
                                             c.c_int, V, V]
        lib.pa_reshape_and_cache.restype = c.c_int
        lib.pa_decode_plan.argtypes = [I32, I32, I32, I32, I32, I32,
                                       c.POINTER(I32), c.POINTER(SZ)]
        lib.pa_decode_plan.restype = c.c_int
        lib.pa_decode.argtypes = [V, I64, V, I64, V, V, V, I64, I32, V, I32, I32, I32, I32,
                                  I32, I64, F, I32, I32, V, SZ, c.c_int, V, V]
        lib.pa_decode.restype = c.c_int
        lib.pa_decode_write.argtypes = [V, I64, V, I64, V, V, I64, V, V, V, I32, V, I64, I32,
                                        V, I32, I32, I32, I32, I32, I64, F, I32, I32, V, SZ,
                                        c.c_int, V, V]
        lib.pa_decode_write.restype = c.c_int
        lib.pa_prefill_varlen.argtypes = [V, I64, V, I64, V, V, V, I64, I32, V, V, I32, I32,
                                          I32, I32, I32, I32, I32, I32, I64, F, I32, c.c_int,
                                          V, V]
        lib.pa_prefill_varlen.restype = c.c_int
        lib.pa_reshape_and_cache_int8.argtypes = [V, V, I64, V, V, V, I32, I32, I32, I32, I64,
                                                  V, V, c.c_int, V, V]
        lib.pa_reshape_and_cache_int8.restype = c.c_int
        lib.pa_copy_blocks.argtypes = [V, V, I64, I64, V, I32, V, V]
        lib.pa_copy_blocks.restype = c.c_int
        lib.pa_decode_int8.argtypes = [V, I64, V, I64, V, V, V, I64, I32, V, I32, I32, I32,
                                       I32, I32, I64, V, V, F, I32, I32, V, SZ, c.c_int, V, V]
        lib.pa_decode_int8.restype = c.c_int
        lib.pa_decode_write_int8.argtypes = [V, I64, V, I64, V, V, I64, V, V, V, I32, V, I64,
                                             I32, V, I32, I32, I32, I32, I32, I64, V, V, F, I32,
                                             I32, V, SZ, c.c_int, V, V]
        lib.pa_decode_write_int8.restype = c.c_int
        lib.pa_reshape_and_cache_fp8.argtypes = lib.pa_reshape_and_cache_int8.argtypes
        lib.pa_reshape_and_cache_fp8.restype = c.c_int
        lib.pa_decode_fp8.argtypes = lib.pa_decode_int8.argtypes
        lib.pa_decode_fp8.restype = c.c_int
        lib.pa_decode_write_fp8.argtypes = lib.pa_decode_write_int8.argtypes
        lib.pa_decode_write_fp8.restype = c.c_int
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int, what: str):
    if status != 0:
        msg = lib.pa_status_string(status).decode()
        if status == 6:
            msg += f" (cudaError {lib.pa_last_cuda_error()})"
        raise PaError(status, f"{what}: {msg}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _rows(t, name):
    """(row stride in elements) of a [rows, heads, head_dim] view with
    contiguous heads."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be [rows, heads, head_dim] with contiguous heads")
    return t.stride(0)


def pa_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, *,
                         d_error=None, stream=None, lib=None):
    """key/value [N, Hkv, D] (equal row strides); caches [NB, bs, Hkv, D]
    contiguous; slot_mapping int64 [N]."""
    lib = lib or library()
    ks = _rows(key, "key")
    if _rows(value, "value") != ks:
        raise ValueError("key and value must share a row stride")
    if not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, D]")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    nb, bs, hkv, d = key_cache.shape
    st = lib.pa_reshape_and_cache(_ptr(key), _ptr(value), ks, _ptr(key_cache),
                                  _ptr(value_cache), _ptr(slot_mapping), key.shape[0], hkv, d,
                                  bs, nb, _DTYPE[key.dtype], _ptr(d_error), _stream(stream))
    _check(lib, st, "pa_reshape_and_cache")


def _scales(t, hkv, what):
    if t.dtype != torch.float32 or t.numel() != hkv or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous float32 tensor of num_kv_heads values")
    return _ptr(t)


_POOL8 = {"int8": (torch.int8,), "fp8": (torch.uint8, torch.float8_e4m3fn)}


def _check_pools8(fmt, key_cache, value_cache):
    if key_cache.dtype not in _POOL8[fmt] or value_cache.dtype not in _POOL8[fmt]:
        names = " or ".join(str(t).replace("torch.", "") for t in _POOL8[fmt])
        raise ValueError(f"{fmt.upper()} caches must be {names}")
    if not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, D]")


def _write8(fmt, key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale, d_error,
            stream, lib):
    lib = lib or library()
    ks = _rows(key, "key")
    if _rows(value, "value") != ks:
        raise ValueError("key and value must share a row stride")
    _check_pools8(fmt, key_cache, value_cache)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    nb, bs, hkv, d = key_cache.shape
    name = f"pa_reshape_and_cache_{fmt}"
    st = getattr(lib, name)(
        _ptr(key), _ptr(value), ks, _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping),
        key.shape[0], hkv, d, bs, nb, _scales(k_scale, hkv, "k_scale"),
        _scales(v_scale, hkv, "v_scale"), _DTYPE[key.dtype], _ptr(d_error), _stream(stream))
    _check(lib, st, name)


def pa_reshape_and_cache_int8(key, value, key_cache, value_cache, slot_mapping, k_scale,
                              v_scale, *, d_error=None, stream=None, lib=None):
    """pa_reshape_and_cache into INT8 pools: caches int8 [NB, bs, Hkv, D];
    k_scale / v_scale float32 [Hkv] (per-KV-head dequantisation scales)."""
    _write8("int8", key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale,
            d_error, stream, lib)


def pa_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale,
                             v_scale, *, d_error=None, stream=None, lib=None):
    """pa_reshape_and_cache into FP8 pools: caches of E4M3 codes (uint8 or
    float8_e4m3fn) [NB, bs, Hkv, D]; k_scale / v_scale float32 [Hkv]."""
    _write8("fp8", key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale,
            d_error, stream, lib)


def pa_copy_blocks(key_cache, value_cache, block_mapping, *, d_error=None, stream=None,
                   lib=None):
    """Copy-on-write of whole blocks: for each row (src, dst) of block_mapping
    (int64 [n, 2] on the device), block dst of both pools receives block src.
    The pools are contiguous [num_blocks, ...] tensors of one shape and dtype
    (16-bit or INT8 pools alike)."""
    lib = lib or library()
    if key_cache.shape != value_cache.shape or key_cache.dtype != value_cache.dtype:
        raise ValueError("key_cache and value_cache must share shape and dtype")
    if not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, ...]")
    if block_mapping.dtype != torch.int64 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous int64 tensor [n, 2]")
    if block_mapping.numel() % 2:
        raise ValueError("block_mapping must hold (src, dst) pairs")
    nb = key_cache.shape[0]
    block_bytes = key_cache.element_size()
    for n in key_cache.shape[1:]:
        block_bytes *= n
    st = lib.pa_copy_blocks(_ptr(key_cache), _ptr(value_cache), block_bytes, nb,
                            _ptr(block_mapping), block_mapping.numel() // 2, _ptr(d_error),
                            _stream(stream))
    _check(lib, st, "pa_copy_blocks")


def pa_debug_set_wait_limit_ns(ns: int, *, lib=None):
    """Bound (ns) of the kernels' pipeline waits for later launches; 0 = the
    default 2 s.  A testing aid: lets a test make waits run out."""
    (lib or library()).pa_debug_set_wait_limit_ns(int(ns))


def pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                   partition_size=0, lib=None):
    """(partition_size, workspace_bytes) that pa_decode will use."""
    lib = lib or library()
    p = ctypes.c_int32(0)
    ws = ctypes.c_size_t(0)
    st = lib.pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                            partition_size, ctypes.byref(p), ctypes.byref(ws))
    _check(lib, st, "pa_decode_plan")
    return p.value, ws.value


def pa_decode(out, query, key_cache, value_cache, block_table, context_lens, *, scale,
              max_context_len, partition_size=0, workspace=None, d_error=None, stream=None,
              lib=None):
    """out/query [S, Hq, D]; caches [NB, bs, Hkv, D]; block_table int32
    [S, max_blocks]; context_lens int32 [S].  ``max_context_len`` is the
    host-side upper bound of context_lens.  A workspace is allocated with
    torch when the plan needs one and none is given."""
    lib = lib or library()
    s, hq, d = query.shape
    nb, bs, hkv, _ = key_cache.shape
    P, need = pa_decode_plan(s, hq, hkv, d, max_context_len, partition_size, lib=lib)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_table and context_lens must be int32")
    st = lib.pa_decode(_ptr(out), _rows(out, "out"), _ptr(query), _rows(query, "query"),
                       _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
                       block_table.stride(0), block_table.shape[1], _ptr(context_lens), s, hq,
                       hkv, d, bs, nb, float(scale), int(max_context_len), P,
                       _ptr(workspace), wbytes, _DTYPE[query.dtype], _ptr(d_error),
                       _stream(stream))
    _check(lib, st, "pa_decode")
    return out


def _decode8(fmt, out, query, key_cache, value_cache, block_table, context_lens, k_scale,
             v_scale, scale, max_context_len, partition_size, workspace, d_error, stream, lib):
    lib = lib or library()
    s, hq, d = query.shape
    nb, bs, hkv, _ = key_cache.shape
    _check_pools8(fmt, key_cache, value_cache)
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_table and context_lens must be int32")
    P, need = pa_decode_plan(s, hq, hkv, d, max_context_len, partition_size, lib=lib)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    name = f"pa_decode_{fmt}"
    st = getattr(lib, name)(
        _ptr(out), _rows(out, "out"), _ptr(query), _rows(query, "query"), _ptr(key_cache),
        _ptr(value_cache), _ptr(block_table), block_table.stride(0), block_table.shape[1],
        _ptr(context_lens), s, hq, hkv, d, bs, nb, _scales(k_scale, hkv, "k_scale"),
        _scales(v_scale, hkv, "v_scale"), float(scale), int(max_context_len), P,
        _ptr(workspace), wbytes, _DTYPE[query.dtype], _ptr(d_error), _stream(stream))
    _check(lib, st, name)
    return out


def pa_decode_int8(out, query, key_cache, value_cache, block_table, context_lens, k_scale,
                   v_scale, *, scale, max_context_len, partition_size=0, workspace=None,
                   d_error=None, stream=None, lib=None):
    """pa_decode over INT8 pools (int8 [NB, bs, Hkv, D], head_dim 64 or 128) with
    per-KV-head float32 scales k_scale / v_scale [Hkv]."""
    return _decode8("int8", out, query, key_cache, value_cache, block_table, context_lens,
                    k_scale, v_scale, scale, max_context_len, partition_size, workspace,
                    d_error, stream, lib)


def pa_decode_fp8(out, query, key_cache, value_cache, block_table, context_lens, k_scale,
                  v_scale, *, scale, max_context_len, partition_size=0, workspace=None,
                  d_error=None, stream=None, lib=None):
    """pa_decode over FP8 pools (E4M3 codes, uint8 or float8_e4m3fn
    [NB, bs, Hkv, D], head_dim 64 or 128) with per-KV-head float32 scales."""
    return _decode8("fp8", out, query, key_cache, value_cache, block_table, context_lens,
                    k_scale, v_scale, scale, max_context_len, partition_size, workspace,
                    d_error, stream, lib)


def pa_decode_write(out, query, key, value, key_cache, value_cache, slot_mapping, block_table,
                    context_lens, *, scale, max_context_len, partition_size=0, workspace=None,
                    d_error=None, stream=None, lib=None):
    """One decode step in one call: pa_reshape_and_cache(key, value, ...,
    slot_mapping) then pa_decode(...), the decode overlapping the write.
    Arguments as for those two functions."""
    lib = lib or library()
    s, hq, d = query.shape
    nb, bs, hkv, _ = key_cache.shape
    ks = _rows(key, "key")
    if _rows(value, "value") != ks:
        raise ValueError("key and value must share a row stride")
    if not key_cache.is_contiguous() or not value_cache.is_contiguous():
        raise ValueError("caches must be contiguous [num_blocks, block_size, Hkv, D]")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_table and context_lens must be int32")
    P, need = pa_decode_plan(s, hq, hkv, d, max_context_len, partition_size, lib=lib)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.pa_decode_write(_ptr(out), _rows(out, "out"), _ptr(query), _rows(query, "query"),
                             _ptr(key), _ptr(value), ks, _ptr(key_cache), _ptr(value_cache),
                             _ptr(slot_mapping), key.shape[0], _ptr(block_table),
                             block_table.stride(0), block_table.shape[1], _ptr(context_lens), s,
                             hq, hkv, d, bs, nb, float(scale), int(max_context_len), P,
                             _ptr(workspace), wbytes, _DTYPE[query.dtype], _ptr(d_error),
                             _stream(stream))
    _check(lib, st, "pa_decode_write")
    return out


def _decode_write8(fmt, out, query, key, value, key_cache, value_cache, slot_mapping,
                   block_table, context_lens, k_scale, v_scale, scale, max_context_len,
                   partition_size, workspace, d_error, stream, lib):
    lib = lib or library()
    s, hq, d = query.shape
    nb, bs, hkv, _ = key_cache.shape
    ks = _rows(key, "key")
    if _rows(value, "value") != ks:
        raise ValueError("key and value must share a row stride")
    _check_pools8(fmt, key_cache, value_cache)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_table and context_lens must be int32")
    P, need = pa_decode_plan(s, hq, hkv, d, max_context_len, partition_size, lib=lib)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    name = f"pa_decode_write_{fmt}"
    st = getattr(lib, name)(
        _ptr(out), _rows(out, "out"), _ptr(query), _rows(query, "query"), _ptr(key),
        _ptr(value), ks, _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping), key.shape[0],
        _ptr(block_table), block_table.stride(0), block_table.shape[1], _ptr(context_lens), s,
        hq, hkv, d, bs, nb, _scales(k_scale, hkv, "k_scale"), _scales(v_scale, hkv, "v_scale"),
        float(scale), int(max_context_len), P, _ptr(workspace), wbytes, _DTYPE[query.dtype],
        _ptr(d_error), _stream(stream))
    _check(lib, st, name)
    return out


def pa_decode_write_int8(out, query, key, value, key_cache, value_cache, slot_mapping,
                         block_table, context_lens, k_scale, v_scale, *, scale, max_context_len,
                         partition_size=0, workspace=None, d_error=None, stream=None, lib=None):
    """One decode step over INT8 pools in one call: pa_reshape_and_cache_int8
    then pa_decode_int8, the decode overlapping the write.  Arguments as for
    those two functions."""
    return _decode_write8("int8", out, query, key, value, key_cache, value_cache, slot_mapping,
                          block_table, context_lens, k_scale, v_scale, scale, max_context_len,
                          partition_size, workspace, d_error, stream, lib)


def pa_decode_write_fp8(out, query, key, value, key_cache, value_cache, slot_mapping,
                        block_table, context_lens, k_scale, v_scale, *, scale, max_context_len,
                        partition_size=0, workspace=None, d_error=None, stream=None, lib=None):
    """One decode step over FP8 pools in one call: pa_reshape_and_cache_fp8
    then pa_decode_fp8.  Arguments as for those two functions."""
    return _decode_write8("fp8", out, query, key, value, key_cache, value_cache, slot_mapping,
                          block_table, context_lens, k_scale, v_scale, scale, max_context_len,
                          partition_size, workspace, d_error, stream, lib)


def pa_prefill_varlen(out, query, key_cache, value_cache, block_table, cu_seqlens_q,
                      context_lens, *, scale, max_seqlen_q, max_context_len, causal=True,
                      d_error=None, stream=None, lib=None):
    """out/query [T, Hq, D] packed by cu_seqlens_q int32 [S+1];
    context_lens int32 [S].  ``max_seqlen_q`` / ``max_context_len`` are host
    upper bounds; T (total_q) is taken from query.shape[0]."""
    lib = lib or library()
    t, hq, d = query.shape
    nb, bs, hkv, _ = key_cache.shape
    s = context_lens.shape[0]
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32 \
            or cu_seqlens_q.dtype != torch.int32:
        raise ValueError("block_table, cu_seqlens_q and context_lens must be int32")
    st = lib.pa_prefill_varlen(_ptr(out), _rows(out, "out"), _ptr(query), _rows(query, "query"),
                               _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
                               block_table.stride(0), block_table.shape[1], _ptr(cu_seqlens_q),
                               _ptr(context_lens), s, t, int(max_seqlen_q),
                               int(max_context_len), hq, hkv, d, bs, nb, float(scale),
                               1 if causal else 0, _DTYPE[query.dtype], _ptr(d_error),
                               _stream(stream))
    _check(lib, st, "pa_prefill_varlen")
    return out
