"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for paged-KV attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it: the two share no code.

Two parts:

* ``pa_oracle.c`` (built into ``libpa_oracle.so``): the write / gather /
  attend statement of the method in fp64 -- see that file's header.
* Pure-Python index helpers that restate the host-side formulas the pages
  print for building ``block_table``, ``slot_mapping``, ``cu_seqlens`` and
  ``actual_seq_lengths`` (the Runner's job on the pages), pinned by the
  pages' worked examples in ``tests/golden/``.

Sources (cited by page and section):
  [SKILL] cannbot-skills "model-infer-kvcache" skill page (devpress.csdn.net)
  [LQNN]  "Paged KV Cache is infrastructure, not a renamed cache" (lqnn.cn)
  [MHPQ]  "Paged KV Cache and Packed Sequence in cann-recipes-infer" (mhpq.cn)
  [VLLM]  "vLLM on CANN" (lnwmold.com)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")

F16, BF16 = 0, 1
OK, ERR_ARG, ERR_SLOT, ERR_BLOCK, ERR_LEN, ERR_NOMEM, ERR_SCALE = range(7)

_lock = threading.Lock()
_lib = None


def build(force: bool = False, out: str | None = None, defines=()) -> str:
    """Compile pa_oracle.c with gcc (fp64, OpenMP).  Returns the .so path.

    ``defines`` lets a test compile a deliberately broken variant of the oracle
    into a separate file (``out``) to check that the pins catch it."""
    target = out or _LIB
    if (not force and not defines and os.path.exists(target)
            and os.path.getmtime(target) >= os.path.getmtime(_SRC)):
        return target
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off"]
    cmd += ["-D" + d for d in defines]
    cmd += [_SRC, "-o", target, "-lm"]
    subprocess.run(cmd, check=True)
    return target


def _bind(lib):
    c = ctypes
    P = c.c_void_p
    lib.pao_f16_to_double.argtypes = [c.c_uint16]
    lib.pao_f16_to_double.restype = c.c_double
    lib.pao_bf16_to_double.argtypes = [c.c_uint16]
    lib.pao_bf16_to_double.restype = c.c_double
    lib.pao_decode_array.argtypes = [P, P, c.c_int64, c.c_int]
    lib.pao_decode_array.restype = None
    lib.pao_max_threads.argtypes = []
    lib.pao_max_threads.restype = c.c_int
    lib.pao_set_threads.argtypes = [c.c_int]
    lib.pao_set_threads.restype = None
    lib.pao_write.argtypes = [P, P, P, P, c.c_int64, P, c.c_int64, c.c_int,
                              c.c_int, c.c_int, c.c_int64]
    lib.pao_write.restype = c.c_int
    lib.pao_copy_blocks.argtypes = [P, P, c.c_int64, c.c_int64, P, c.c_int64]
    lib.pao_copy_blocks.restype = c.c_int
    lib.pao_decode.argtypes = [P, P, c.c_int64, P, P, P, c.c_int64, c.c_int,
                               P, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                               c.c_int64, c.c_double, c.c_int]
    lib.pao_decode.restype = c.c_int
    lib.pao_quantize_int8.argtypes = [P, P, c.c_int64, c.c_int, c.c_float]
    lib.pao_quantize_int8.restype = c.c_int
    lib.pao_write_int8.argtypes = [P, P, P, P, c.c_int64, P, c.c_int64, c.c_int,
                                   c.c_int, c.c_int, c.c_int64, c.c_int, P, P]
    lib.pao_write_int8.restype = c.c_int
    lib.pao_decode_int8.argtypes = [P, P, c.c_int64, P, P, P, c.c_int64, c.c_int,
                                    P, c.c_int, c.c_int, c.c_int, c.c_int, c.c_int,
                                    c.c_int64, c.c_double, c.c_int, P, P]
    lib.pao_decode_int8.restype = c.c_int
    lib.pao_fp8_value.argtypes = [P, P, c.c_int64]
    lib.pao_fp8_value.restype = None
    lib.pao_quantize_fp8.argtypes = [P, P, c.c_int64, c.c_int, c.c_float]
    lib.pao_quantize_fp8.restype = c.c_int
    lib.pao_write_fp8.argtypes = lib.pao_write_int8.argtypes
    lib.pao_write_fp8.restype = c.c_int
    lib.pao_decode_fp8.argtypes = lib.pao_decode_int8.argtypes
    lib.pao_decode_fp8.restype = c.c_int
    lib.pao_prefill.argtypes = [P, P, c.c_int64, P, P, P, c.c_int64, c.c_int,
                                P, P, c.c_int, c.c_int64, c.c_int, c.c_int,
                                c.c_int, c.c_int, c.c_int64, c.c_double,
                                c.c_int, P, c.c_int]
    lib.pao_prefill.restype = c.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _u16(a) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 torch tensor or a uint16 array."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch
    assert a.dtype in (torch.float16, torch.bfloat16), a.dtype
    return np.ascontiguousarray(
        a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def dtype_code(torch_dtype) -> int:
    import torch
    return BF16 if torch_dtype == torch.bfloat16 else F16


def set_threads(n: int, lib=None) -> None:
    (lib or load()).pao_set_threads(int(n))


def max_threads(lib=None) -> int:
    return int((lib or load()).pao_max_threads())


def decode16(patterns: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """fp64 values of 16-bit patterns, decoded by the oracle's own decoder."""
    lib = lib or load()
    p = np.ascontiguousarray(patterns, dtype=np.uint16)
    out = np.empty(p.shape, dtype=np.float64)
    lib.pao_decode_array(_ptr(out), _ptr(p), p.size, int(dtype))
    return out


def write(k_pool: np.ndarray, v_pool: np.ndarray, k_new, v_new, slot_mapping,
          block_size: int, lib=None) -> int:
    """Apply the cache write in place on uint16 pools [NB, bs, Hkv, D].

    ``k_new``/``v_new``: [N, Hkv, D] fp16/bf16 tensors or uint16 arrays.
    Returns the oracle status (OK, or ERR_SLOT if a slot was out of range;
    out-of-range rows are skipped)."""
    lib = lib or load()
    kn, vn = _u16(k_new), _u16(v_new)
    n = kn.shape[0]
    hkv, d = kn.shape[1], kn.shape[2]
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
    nb = k_pool.shape[0]
    return lib.pao_write(_ptr(k_pool), _ptr(v_pool), _ptr(kn), _ptr(vn),
                         hkv * d, _ptr(slots), n, hkv, d, block_size, nb)



def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, block_mapping, lib=None) -> int:
    """Copy-on-write of whole blocks in place: for each (src, dst) row of
    block_mapping (int [n, 2]), block dst of both pools receives block src,
    byte for byte, in order.  Pools are C-contiguous numpy arrays
    [num_blocks, ...] of any dtype.  Returns OK, or ERR_BLOCK if a pair named
    a block outside the pool (that pair copies nothing)."""
    lib = lib or load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.shape == v_pool.shape and k_pool.dtype == v_pool.dtype
    bm = np.ascontiguousarray(np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2))
    nb = k_pool.shape[0]
    block_bytes = k_pool.nbytes // nb if nb else 0
    if nb == 0:
        return OK if bm.shape[0] == 0 else ERR_BLOCK
    return lib.pao_copy_blocks(_ptr(k_pool), _ptr(v_pool), block_bytes, nb, _ptr(bm),
                               bm.shape[0])

def decode(q, k_pool, v_pool, block_table, context_lens, num_kv_heads: int,
           block_size: int, scale: float, dtype: int | None = None,
           lib=None, return_status: bool = False):
    """Oracle decode.  q: [S, Hq, D]; pools: [NB, bs, Hkv, D]; block_table:
    [S, max_blocks] int32; context_lens: [S] int32.  Returns fp64 [S, Hq, D]."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(q.dtype)
    qu, ku, vu = _u16(q), _u16(k_pool), _u16(v_pool)
    bt = np.ascontiguousarray(np.asarray(block_table), dtype=np.int32)
    ctx = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    s, hq, d = qu.shape
    nb = ku.shape[0]
    out = np.zeros((s, hq, d), dtype=np.float64)
    st = lib.pao_decode(_ptr(out), _ptr(qu), hq * d, _ptr(ku), _ptr(vu),
                        _ptr(bt), bt.shape[1], bt.shape[1], _ptr(ctx), s, hq,
                        num_kv_heads, d, block_size, nb, float(scale), dtype)
    return (out, st) if return_status else out


def quantize_int8(x, scale: float, dtype: int | None = None, lib=None,
                  return_status: bool = False):
    """INT8 codes of fp16/bf16 values (a tensor, or uint16 patterns with
    ``dtype``) under one scale: round-half-even(x / scale) in fp32, clamped
    to [-127, 127]."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(x.dtype)
    xu = _u16(x)
    codes = np.zeros(xu.shape, dtype=np.int8)
    st = lib.pao_quantize_int8(_ptr(codes), _ptr(xu), xu.size, int(dtype),
                               float(np.float32(scale)))
    return (codes, st) if return_status else codes


def _scales(a, n: int) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(a, dtype=np.float32).reshape(-1))
    assert v.size == n, (v.size, n)
    return v


def write_int8(k_pool: np.ndarray, v_pool: np.ndarray, k_new, v_new, slot_mapping,
               block_size: int, k_scale, v_scale, dtype: int | None = None,
               lib=None) -> int:
    """The cache write into INT8 pools [NB, bs, Hkv, D], quantising each new
    row per KV head with k_scale / v_scale ([Hkv] fp32).  Returns the status."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(k_new.dtype)
    kn, vn = _u16(k_new), _u16(v_new)
    n, hkv, d = kn.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_pool.dtype == np.int8 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.int8 and v_pool.flags.c_contiguous
    ks, vs = _scales(k_scale, hkv), _scales(v_scale, hkv)
    return lib.pao_write_int8(_ptr(k_pool), _ptr(v_pool), _ptr(kn), _ptr(vn),
                              hkv * d, _ptr(slots), n, hkv, d, block_size,
                              k_pool.shape[0], int(dtype), _ptr(ks), _ptr(vs))


def decode_int8(q, k_pool: np.ndarray, v_pool: np.ndarray, block_table, context_lens,
                num_kv_heads: int, block_size: int, scale: float, k_scale, v_scale,
                dtype: int | None = None, lib=None, return_status: bool = False):
    """Oracle decode over INT8 pools ([NB, bs, Hkv, D] int8, dequantised per
    KV head).  Returns fp64 [S, Hq, D]."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(q.dtype)
    qu = _u16(q)
    ku = np.ascontiguousarray(k_pool, dtype=np.int8)
    vu = np.ascontiguousarray(v_pool, dtype=np.int8)
    bt = np.ascontiguousarray(np.asarray(block_table), dtype=np.int32)
    ctx = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    s, hq, d = qu.shape
    ks, vs = _scales(k_scale, num_kv_heads), _scales(v_scale, num_kv_heads)
    out = np.zeros((s, hq, d), dtype=np.float64)
    st = lib.pao_decode_int8(_ptr(out), _ptr(qu), hq * d, _ptr(ku), _ptr(vu), _ptr(bt),
                             bt.shape[1], bt.shape[1], _ptr(ctx), s, hq, num_kv_heads,
                             d, block_size, ku.shape[0], float(scale), dtype,
                             _ptr(ks), _ptr(vs))
    return (out, st) if return_status else out


def fp8_value(codes, lib=None) -> np.ndarray:
    """Values (fp64) of FP8 E4M3 codes (uint8), from the format's definition."""
    lib = lib or load()
    cu = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(cu.shape, dtype=np.float64)
    lib.pao_fp8_value(_ptr(out), _ptr(cu), cu.size)
    return out


def quantize_fp8(x, scale: float, dtype: int | None = None, lib=None,
                 return_status: bool = False):
    """FP8 E4M3 codes (uint8) of fp16/bf16 values under one scale: the nearest
    E4M3 value to x / scale (fp32 division; ties to even; saturating at
    448); NaN -> 0."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(x.dtype)
    xu = _u16(x)
    codes = np.zeros(xu.shape, dtype=np.uint8)
    st = lib.pao_quantize_fp8(_ptr(codes), _ptr(xu), xu.size, int(dtype),
                              float(np.float32(scale)))
    return (codes, st) if return_status else codes


def write_fp8(k_pool: np.ndarray, v_pool: np.ndarray, k_new, v_new, slot_mapping,
              block_size: int, k_scale, v_scale, dtype: int | None = None,
              lib=None) -> int:
    """The cache write into FP8 pools [NB, bs, Hkv, D] (uint8 E4M3 codes),
    quantising each new row per KV head.  Returns the status."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(k_new.dtype)
    kn, vn = _u16(k_new), _u16(v_new)
    n, hkv, d = kn.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous
    assert v_pool.dtype == np.uint8 and v_pool.flags.c_contiguous
    ks, vs = _scales(k_scale, hkv), _scales(v_scale, hkv)
    return lib.pao_write_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(kn), _ptr(vn),
                             hkv * d, _ptr(slots), n, hkv, d, block_size,
                             k_pool.shape[0], int(dtype), _ptr(ks), _ptr(vs))


def decode_fp8(q, k_pool: np.ndarray, v_pool: np.ndarray, block_table, context_lens,
               num_kv_heads: int, block_size: int, scale: float, k_scale, v_scale,
               dtype: int | None = None, lib=None, return_status: bool = False):
    """Oracle decode over FP8 pools ([NB, bs, Hkv, D] uint8 E4M3 codes,
    dequantised per KV head).  Returns fp64 [S, Hq, D]."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(q.dtype)
    qu = _u16(q)
    ku = np.ascontiguousarray(k_pool, dtype=np.uint8)
    vu = np.ascontiguousarray(v_pool, dtype=np.uint8)
    bt = np.ascontiguousarray(np.asarray(block_table), dtype=np.int32)
    ctx = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    s, hq, d = qu.shape
    ks, vs = _scales(k_scale, num_kv_heads), _scales(v_scale, num_kv_heads)
    out = np.zeros((s, hq, d), dtype=np.float64)
    st = lib.pao_decode_fp8(_ptr(out), _ptr(qu), hq * d, _ptr(ku), _ptr(vu), _ptr(bt),
                            bt.shape[1], bt.shape[1], _ptr(ctx), s, hq, num_kv_heads,
                            d, block_size, ku.shape[0], float(scale), dtype,
                            _ptr(ks), _ptr(vs))
    return (out, st) if return_status else out


def prefill(q, k_pool, v_pool, block_table, cu_seqlens_q, context_lens,
            num_kv_heads: int, block_size: int, scale: float,
            causal: bool = True, rows=None, dtype: int | None = None,
            lib=None, return_status: bool = False):
    """Oracle varlen prefill.  q: [T, Hq, D] packed by cu_seqlens_q [S+1];
    ``rows`` optionally restricts the computed packed rows (others are NaN).
    Returns fp64 [T, Hq, D]."""
    lib = lib or load()
    if dtype is None:
        dtype = dtype_code(q.dtype)
    qu, ku, vu = _u16(q), _u16(k_pool), _u16(v_pool)
    bt = np.ascontiguousarray(np.asarray(block_table), dtype=np.int32)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_q), dtype=np.int32)
    ctx = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    t, hq, d = qu.shape
    nb = ku.shape[0]
    mask = None
    out = np.zeros((t, hq, d), dtype=np.float64)
    if rows is not None:
        mask = np.zeros(t, dtype=np.uint8)
        mask[np.asarray(rows, dtype=np.int64)] = 1
        out[:] = np.nan
    st = lib.pao_prefill(_ptr(out), _ptr(qu), hq * d, _ptr(ku), _ptr(vu),
                         _ptr(bt), bt.shape[1], bt.shape[1], _ptr(cu),
                         _ptr(ctx), len(ctx), t, hq, num_kv_heads, d,
                         block_size, nb, float(scale), int(bool(causal)),
                         _ptr(mask), dtype)
    return (out, st) if return_status else out


# ---------------------------------------------------------------------------
# Host-side index formulas (the Runner's side of the pages), pure Python.
# ---------------------------------------------------------------------------

def slot_of(block_table, batch_idx: int, seq_pos: int, block_size: int) -> int:
    """Physical slot of (batch_idx, seq_pos): logical block seq_pos //
    block_size, offset seq_pos % block_size, physical block from the block
    table, slot = block * block_size + offset ([SKILL] §3.1 mapping formula)."""
    logical_block = seq_pos // block_size
    offset = seq_pos % block_size
    physical = int(block_table[batch_idx][logical_block])
    return physical * block_size + offset


def static_block_table(batch_size: int, max_seq_len: int, block_size: int):
    """The pre-allocated table that stays fixed for the whole inference:
    row b holds blocks b*n .. b*n+n-1 with n = max_seq_len // block_size
    ([SKILL] §3.2)."""
    n = max_seq_len // block_size
    return [[b * n + i for i in range(n)] for b in range(batch_size)]


def sequential_prefill_slots(kv_len, max_seq_len: int):
    """Prefill slot_mapping in the sequential pool: batch b writes slots
    b*max_seq_len .. b*max_seq_len + kv_len[b] - 1, concatenated
    ([SKILL] §3.3, prefill)."""
    out = []
    for b, n in enumerate(kv_len):
        out.extend(range(b * max_seq_len, b * max_seq_len + int(n)))
    return out


def sequential_decode_slots(kv_len, max_seq_len: int):
    """Decode slot_mapping: one slot per batch, kv_len[b] + b*max_seq_len
    ([SKILL] §3.3, decode)."""
    return [[int(n) + b * max_seq_len] for b, n in enumerate(kv_len)]


def cu_seqlens(lengths):
    """cu_seqlens[0] = 0, cu_seqlens[i+1] = cu_seqlens[i] + lengths[i];
    length batch+1, last entry the packed total ([LQNN] §3.1, §3.3)."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def tnd_actual_seq_lengths(lengths):
    """TND layout passes cumulative lengths without the leading 0
    ([SKILL] §3.4)."""
    return cu_seqlens(lengths)[1:]


def decode_context_lens(kv_len):
    """After writing the new token at position kv_len, attention must read
    kv_len + 1 keys ([SKILL] §3.6: actual_seq_lengths_kv = kv_len + 1)."""
    return [int(n) + 1 for n in kv_len]


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(num_tokens / block_size) ([VLLM] allocate_slots; [LQNN] §2.2)."""
    return (int(num_tokens) + block_size - 1) // block_size
