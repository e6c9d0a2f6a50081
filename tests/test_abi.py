"""The C-ABI library loads, exports every entry point include/pa.h declares,
and rejects bad arguments on the host before touching the GPU.  These calls
return before any CUDA call, so they run without a GPU."""
import ctypes
import os
import re

import pytest
import torch  # noqa: F401  (loads the CUDA runtime libpa.so links against)

import paged_kv_cache_34_gb300 as pa
from paged_kv_cache_34_gb300 import build as pabuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    pabuild.build()
    return pa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pa_reshape_and_cache", "pa_decode", "pa_prefill_varlen"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"


def test_abi_version_matches_header(lib):
    m = re.search(r"#define PA_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.pa_abi_version() == int(m.group(1))


def test_status_strings(lib):
    for code, name in pa._STATUS.items():
        assert lib.pa_status_string(code).decode().startswith(name)


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def decode_call(lib, **kw):
    a = dict(out=FAKE, out_stride=8 * 128, q=FAKE, q_stride=8 * 128, kc=FAKE, vc=FAKE,
             bt=FAKE, bt_stride=16, mbps=16, ctx=FAKE, s=4, hq=8, hkv=2, d=128, bs=16,
             nb=64, scale=0.125, maxctx=100, part=0, ws=None, wsb=0, dtype=0)
    a.update(kw)
    return lib.pa_decode(a["out"], a["out_stride"], a["q"], a["q_stride"], a["kc"], a["vc"],
                         a["bt"], a["bt_stride"], a["mbps"], a["ctx"], a["s"], a["hq"],
                         a["hkv"], a["d"], a["bs"], a["nb"], a["scale"], a["maxctx"],
                         a["part"], a["ws"], a["wsb"], a["dtype"], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(hkv=3), 2),                       # Hq % Hkv != 0
    (dict(hq=8, hkv=16), 2),                # more KV heads than query heads
    (dict(d=96), 3),                        # head_dim not built
    (dict(bs=24), 3),                       # block size not built
    (dict(bt_stride=8), 2),                 # stride < max_blocks_per_seq
    (dict(part=100), 2),                    # partition not a multiple of 64
    (dict(scale=float("nan")), 2),          # scale must be finite
    (dict(dtype=7), 3),
    (dict(q=None), 1),
    (dict(q_stride=8 * 128 - 8), 2),        # row stride below Hq*D
    (dict(q_stride=8 * 128 + 4), 4),        # row stride not a multiple of 8
    (dict(kc=MISALIGNED), 4),
    (dict(s=-1), 2),
])
def test_decode_host_validation(lib, kw, status):
    assert decode_call(lib, **kw) == status


def test_decode_empty_batch_is_ok(lib):
    assert decode_call(lib, s=0) == 0


def prefill_call(lib, **kw):
    a = dict(out=FAKE, q=FAKE, stride=32 * 128, kc=FAKE, vc=FAKE, bt=FAKE, bt_stride=16,
             mbps=16, cu=FAKE, ctx=FAKE, s=2, t=100, maxq=64, maxctx=64, hq=32, hkv=32,
             d=128, bs=128, nb=64, scale=0.088, causal=1, dtype=1)
    a.update(kw)
    return lib.pa_prefill_varlen(a["out"], a["stride"], a["q"], a["stride"], a["kc"], a["vc"],
                                 a["bt"], a["bt_stride"], a["mbps"], a["cu"], a["ctx"], a["s"],
                                 a["t"], a["maxq"], a["maxctx"], a["hq"], a["hkv"], a["d"],
                                 a["bs"], a["nb"], a["scale"], a["causal"], a["dtype"], None,
                                 None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=96), 3), (dict(bs=8), 3), (dict(hkv=5), 2), (dict(cu=None), 1),
    (dict(out=MISALIGNED), 4), (dict(t=-1), 2), (dict(nb=0), 2),
])
def test_prefill_host_validation(lib, kw, status):
    assert prefill_call(lib, **kw) == status


def test_prefill_empty_is_ok(lib):
    assert prefill_call(lib, t=0) == 0 and prefill_call(lib, s=0) == 0


def test_reshape_host_validation(lib):
    f = lib.pa_reshape_and_cache
    # zero tokens: nothing to do
    assert f(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 0, 2, 64, 16, 8, 0, None, None) == 0
    assert f(None, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 0, None, None) == 1
    assert f(FAKE, FAKE, 100, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 0, None, None) == 2
    assert f(FAKE, FAKE, 260, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 0, None, None) == 4
    assert f(FAKE, MISALIGNED, 256, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 0, None, None) == 4
    assert f(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 64, 16, 8, 5, None, None) == 3


def decode_write_call(lib, **kw):
    a = dict(out=FAKE, q=FAKE, q_stride=8 * 128, k=FAKE, v=FAKE, kv_stride=2 * 128, kc=FAKE,
             vc=FAKE, slots=FAKE, n=4, bt=FAKE, bt_stride=16, mbps=16, ctx=FAKE, s=4, hq=8,
             hkv=2, d=128, bs=16, nb=64, scale=0.125, maxctx=100, part=0, dtype=0)
    a.update(kw)
    return lib.pa_decode_write(a["out"], a["q_stride"], a["q"], a["q_stride"], a["k"], a["v"],
                               a["kv_stride"], a["kc"], a["vc"], a["slots"], a["n"], a["bt"],
                               a["bt_stride"], a["mbps"], a["ctx"], a["s"], a["hq"], a["hkv"],
                               a["d"], a["bs"], a["nb"], a["scale"], a["maxctx"], a["part"],
                               None, 0, a["dtype"], None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(kv_stride=100), 2),      # the write's row stride is below Hkv*D
    (dict(slots=None), 1),         # the write's slot_mapping is missing
    (dict(k=MISALIGNED), 4),       # the write's key is misaligned
    (dict(hkv=3), 2),              # the decode's Hq % Hkv != 0
    (dict(d=96), 3),               # the decode's head_dim is not built
    (dict(q=None), 1),             # the decode's query is missing
    (dict(part=100), 2),           # the decode's partition is not a multiple of 16
])
def test_decode_write_checks_both_halves_before_enqueueing(lib, kw, status):
    # every case fails on the host, before any CUDA call
    assert decode_write_call(lib, **kw) == status


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        pa.library(str(tmp_path / "libpa.so"))


def decode_int8_call(lib, **kw):
    a = dict(out=FAKE, out_stride=8 * 128, q=FAKE, q_stride=8 * 128, kc=FAKE, vc=FAKE,
             bt=FAKE, bt_stride=16, mbps=16, ctx=FAKE, s=4, hq=8, hkv=2, d=128, bs=16,
             nb=64, ks=FAKE, vs=FAKE, scale=0.125, maxctx=100, part=0, dtype=1)
    a.update(kw)
    return lib.pa_decode_int8(a["out"], a["out_stride"], a["q"], a["q_stride"], a["kc"],
                              a["vc"], a["bt"], a["bt_stride"], a["mbps"], a["ctx"], a["s"],
                              a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["ks"], a["vs"],
                              a["scale"], a["maxctx"], a["part"], None, 0, a["dtype"], None,
                              None)


@pytest.mark.parametrize("kw,status", [
    (dict(ks=None), 1),                     # the per-head scales are required
    (dict(vs=None), 1),
    (dict(ks=ctypes.c_void_p(0x10002)), 4),  # scales are fp32: 4-byte aligned
    (dict(d=96), 3),                        # head_dim not built
    (dict(hkv=3), 2),                       # Hq % Hkv != 0
    (dict(kc=MISALIGNED), 4),
    (dict(q=None), 1),
])
def test_decode_int8_host_validation(lib, kw, status):
    assert decode_int8_call(lib, **kw) == status


def test_reshape_int8_host_validation(lib):
    f = lib.pa_reshape_and_cache_int8
    # key, value, stride, k_cache, v_cache, slots, n, hkv, d, bs, nb, k_scale, v_scale, dtype
    assert f(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, FAKE, FAKE, 0, None, None) == 0
    assert f(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 128, 16, 8, None, FAKE, 0, None, None) == 1
    assert f(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 128, 16, 8, FAKE,
             ctypes.c_void_p(0x10002), 0, None, None) == 4
    # head_dim 40: 16-bit rows are fine, but an int8 pool row chunk would span heads
    assert f(FAKE, FAKE, 80, FAKE, FAKE, FAKE, 3, 2, 40, 16, 8, FAKE, FAKE, 0, None, None) == 4
    assert f(None, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 128, 16, 8, FAKE, FAKE, 0, None, None) == 1


def test_copy_blocks_host_validation(lib):
    f = lib.pa_copy_blocks
    # k_cache, v_cache, block_bytes, num_blocks, block_mapping, num_pairs, d_error, stream
    assert f(FAKE, FAKE, 4096, 64, FAKE, 0, None, None) == 0  # nothing to copy
    assert f(FAKE, FAKE, 4096, 64, None, 0, None, None) == 0
    assert f(None, FAKE, 4096, 64, FAKE, 3, None, None) == 1
    assert f(FAKE, FAKE, 4096, 64, None, 3, None, None) == 1
    assert f(FAKE, FAKE, 0, 64, FAKE, 3, None, None) == 2
    assert f(FAKE, FAKE, 4096, -1, FAKE, 3, None, None) == 2
    assert f(FAKE, FAKE, 4096, 64, FAKE, -1, None, None) == 2
    assert f(FAKE, FAKE, 4100, 64, FAKE, 3, None, None) == 4
    assert f(MISALIGNED, FAKE, 4096, 64, FAKE, 3, None, None) == 4
    assert f(FAKE, FAKE, 4096, 64, ctypes.c_void_p(0x10004), 3, None, None) == 4


def test_decode_write_int8_host_validation(lib):
    f = lib.pa_decode_write_int8

    def call(ks=FAKE, vs=FAKE, slots=FAKE, n=4, d=128, kv_stride=2 * 128):
        return f(FAKE, 8 * 128, FAKE, 8 * 128, FAKE, FAKE, kv_stride, FAKE, FAKE, slots, n, FAKE,
                 16, 16, FAKE, 4, 8, 2, d, 16, 64, ks, vs, 0.125, 100, 0, None, 0, 0, None,
                 None)
    assert call(ks=None) == 1
    assert call(vs=None) == 1
    assert call(slots=None) == 1          # the write half is checked first
    assert call(kv_stride=100) == 2
    assert call(d=96, kv_stride=192) == 3  # head_dim not built
    assert call(ks=ctypes.c_void_p(0x10002)) == 4


def test_fp8_host_validation(lib):
    # the FP8 calls share the INT8 calls' checks
    w = lib.pa_reshape_and_cache_fp8
    assert w(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 0, 2, 128, 16, 8, FAKE, FAKE, 0, None, None) == 0
    assert w(FAKE, FAKE, 256, FAKE, FAKE, FAKE, 3, 2, 128, 16, 8, None, FAKE, 0, None, None) == 1
    assert w(FAKE, FAKE, 80, FAKE, FAKE, FAKE, 3, 2, 40, 16, 8, FAKE, FAKE, 0, None, None) == 4
    d = lib.pa_decode_fp8
    # out, out_stride, q, q_stride, kc, vc, bt, bt_stride, mbps, ctx, s, hq, hkv, d, bs, nb,
    # k_scale, v_scale, scale, max_ctx, part, ws, ws_bytes, dtype, err, stream
    assert d(FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, 16, 16, FAKE, 4, 8, 2, 128, 16, 64,
             None, FAKE, 0.125, 100, 0, None, 0, 0, None, None) == 1
    assert d(FAKE, 768, FAKE, 768, FAKE, FAKE, FAKE, 16, 16, FAKE, 4, 8, 2, 96, 16, 64,
             FAKE, FAKE, 0.125, 100, 0, None, 0, 0, None, None) == 3
    s = lib.pa_decode_write_fp8
    assert s(FAKE, 1024, FAKE, 1024, FAKE, FAKE, 256, FAKE, FAKE, None, 4, FAKE, 16, 16, FAKE,
             4, 8, 2, 128, 16, 64, FAKE, FAKE, 0.125, 100, 0, None, 0, 0, None, None) == 1
