"""The pins must be strong enough to catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of the oracle's C source (on the
CPU, in a temporary directory), builds it, and checks that at least one pin
fails for it while the unmodified oracle passes them all."""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_34_gb300 import workloads as W

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    "logical_block_uses_modulo": ("int logical_block = j / block_size;",
                                  "int logical_block = j % block_size;"),
    "offset_uses_division": ("int offset = j % block_size;",
                             "int offset = j / block_size;"),
    "kv_head_ignored": ("+ offset) * hkv + g) * d;", "+ offset) * hkv + 0) * d;"),
    "value_read_from_key_pool": ("vc[(int64_t)j * d + x] = decode16(v_pool",
                                 "vc[(int64_t)j * d + x] = decode16(k_pool"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "no_normalisation": ("o[x] = acc / denom;", "o[x] = acc;"),
    "max_not_subtracted": ("s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
    "causal_top_left": ("int n = causal ? len - qlen + i + 1 : len;",
                        "int n = causal ? i + 1 : len;"),
    "causal_off_by_one": ("int n = causal ? len - qlen + i + 1 : len;",
                          "int n = causal ? len - qlen + i : len;"),
    "f16_exponent_bias": ("v = ldexp((double)(0x400 | f), e - 25);",
                          "v = ldexp((double)(0x400 | f), e - 24);"),
    "bf16_subnormal_scale": ("v = ldexp((double)f, -133);",
                             "v = ldexp((double)f, -126);"),
    "write_offset_swapped": ("int64_t offset = slot % block_size; /* position in block   */",
                             "int64_t offset = slot / block_size;"),
    "int8_round_half_away": ("return (int8_t)rintf(y);", "return (int8_t)roundf(y);"),
    "int8_clamp_late": ("if (y >= 127.0f) return 127;", "if (y >= 128.0f) return 127;"),
    "int8_value_uses_key_scale": ("(double)v_pool[base + x] * v_scale;",
                                  "(double)v_pool[base + x] * k_scale;"),
    "int8_decode_head0_scale": ("block_size, num_blocks, k_scale[g], v_scale[g]);",
                                "block_size, num_blocks, k_scale[0], v_scale[0]);"),
    "int8_write_head0_scale": ("const float ks = k_scale[g], vs = v_scale[g];",
                               "const float ks = k_scale[0], vs = v_scale[0];"),
    "copy_blocks_direction_swapped": (
        "memmove(k_pool + dst * block_bytes, k_pool + src * block_bytes,",
        "memmove(k_pool + src * block_bytes, k_pool + dst * block_bytes,"),
    "copy_blocks_value_skipped": ("memmove(v_pool + dst * block_bytes, v_pool + src",
                                  "(void)(v_pool + dst * block_bytes, v_pool + src"),
    "copy_blocks_half_block": ("k_pool + src * block_bytes,\n            (size_t)block_bytes);",
                               "k_pool + src * block_bytes,\n            (size_t)block_bytes / 2);"),
    "copy_blocks_stops_at_bad_pair": ("      status = PAO_ERR_BLOCK;\n      continue;",
                                      "      status = PAO_ERR_BLOCK;\n      break;"),
    "fp8_exponent_bias": ("else v = ldexp(1.0 + m / 8.0, e - 7);",
                          "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "fp8_subnormal_scale": ("if (e == 0) v = ldexp(m / 8.0, -6);",
                            "if (e == 0) v = ldexp(m / 8.0, -7);"),
    "fp8_ties_away_from_zero": ("((lo & 1) == 0 ? lo : hi)", "(hi)"),
    "fp8_decode_reads_int8": ("= value[k_pool[base + x]] * k_scale;",
                              "= (double)(int8_t)k_pool[base + x] * k_scale;"),
    "decode_heads_strided": (
        "for (int h = g * group; h < (g + 1) * group; ++h) {\n      double *o = out + ((int64_t)b * hq + h) * d;",
        "for (int h = g; h < hq; h += hkv) {\n      double *o = out + ((int64_t)b * hq + h) * d;"),
}


def _build(tmp, name, replace):
    src = open(SRC).read()
    if replace is not None:
        old, new = replace
        assert src.count(old) >= 1, f"mutation site for {name} not found"
        src = src.replace(old, new)
    path = os.path.join(tmp, f"{name}.c")
    open(path, "w").write(src)
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", path, "-o", so, "-lm"], check=True)
    return oracle.load(so)


def _cfg(kind, hq, hkv, d, bs, nb, lengths, placement, dtype="f16"):
    return dict(kind=kind, num_seqs=len(lengths), lengths=("list", lengths, None),
                num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                num_blocks=nb, placement=placement, dtype=dtype, name="m")


def _contig(pool, x, b):
    L = int(x.context_lens[b])
    start = int(x.block_table[b, 0]) * x.block_size
    flat = pool.reshape(-1, x.num_kv_heads, x.head_dim)
    return flat[start:start + L].double().permute(1, 0, 2)


def _pin_decode_sdpa(lib):
    x = W.make_inputs(_cfg("decode", 8, 2, 64, 16, 40, [1, 40, 99],
                           "identity"), seed=31)
    out = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table,
                        x.context_lens, 2, 16, x.scale, lib=lib)
    for b in range(3):
        k, v = _contig(x.k_pool, x, b), _contig(x.v_pool, x, b)
        want = F.scaled_dot_product_attention(
            x.q[b].double()[None, :, None], k[None], v[None], scale=x.scale,
            enable_gqa=True)[0, :, 0]
        if not np.allclose(out[b], want.numpy(), rtol=1e-10, atol=1e-12):
            return False
    return True


def _pin_prefill_sdpa(lib):
    x = W.make_inputs(_cfg("prefill", 4, 2, 64, 16, 40, [33, 70], "identity"),
                      seed=37)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, 16, lib=lib)
    out = oracle.prefill(x.q, kp, vp, x.block_table, x.cu_seqlens_q,
                         x.context_lens, 2, 16, x.scale, dtype=oracle.F16,
                         lib=lib)
    kt = torch.from_numpy(kp.view(np.int16)).view(torch.float16)
    vt = torch.from_numpy(vp.view(np.int16)).view(torch.float16)
    cu = x.cu_seqlens_q.tolist()
    for b in range(2):
        k, v = _contig(kt, x, b), _contig(vt, x, b)
        q = x.q[cu[b]:cu[b + 1]].double().permute(1, 0, 2)
        want = F.scaled_dot_product_attention(q[None], k[None], v[None],
                                              is_causal=True, scale=x.scale,
                                              enable_gqa=True)[0]
        if not np.allclose(out[cu[b]:cu[b + 1]], want.permute(1, 0, 2).numpy(),
                           rtol=1e-10, atol=1e-12):
            return False
    return True


def _pin_chunked_tail(lib):
    # q < L rows must equal the tail rows of SDPA's full causal attention
    x = W.make_inputs(_cfg("prefill", 4, 4, 64, 16, 40, [50], "identity"),
                      seed=41)
    kp = oracle._u16(x.k_pool).copy()
    vp = oracle._u16(x.v_pool).copy()
    oracle.write(kp, vp, x.k_new, x.v_new, x.slot_mapping, 16, lib=lib)
    qn = 9
    out = oracle.prefill(x.q[-qn:], kp, vp, x.block_table, [0, qn],
                         x.context_lens, 4, 16, x.scale, dtype=oracle.F16,
                         lib=lib)
    kt = torch.from_numpy(kp.view(np.int16)).view(torch.float16)
    vt = torch.from_numpy(vp.view(np.int16)).view(torch.float16)
    k, v = _contig(kt, x, 0), _contig(vt, x, 0)
    want = F.scaled_dot_product_attention(
        x.q.double().permute(1, 0, 2)[None], k[None], v[None], is_causal=True,
        scale=x.scale)[0].permute(1, 0, 2)[-qn:]
    return np.allclose(out, want.numpy(), rtol=1e-10, atol=1e-12)


def _pin_decoders(lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.decode16(pats, oracle.F16, lib=lib)
    bf = oracle.decode16(pats, oracle.BF16, lib=lib)
    want16 = pats.view(np.float16).astype(np.float64)
    wantbf = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    return (np.array_equal(f16, want16, equal_nan=True)
            and np.array_equal(bf, wantbf, equal_nan=True))


def _pin_write(lib):
    nb, bs, hkv, d = 4, 8, 1, 2
    kp = np.zeros((nb, bs, hkv, d), np.uint16)
    vp = np.zeros((nb, bs, hkv, d), np.uint16)
    kn = np.array([[[5, 6]]], np.uint16)
    oracle.write(kp, vp, kn, kn, np.array([2 * bs + 3]), bs, lib=lib)
    return kp[2, 3, 0].tolist() == [5, 6] and int(kp.sum()) == 11


def _pin_saturated_softmax(lib):
    # With a huge scale the softmax is one-hot at the best key, so the output
    # is that key's value row (the limit of the closed form).
    x = W.make_inputs(_cfg("decode", 2, 2, 64, 16, 20, [60, 90], "identity"),
                      seed=43)
    big = 1.0e4
    out = oracle.decode(x.q, x.k_pool, x.v_pool, x.block_table,
                        x.context_lens, 2, 16, big, lib=lib)
    for b in range(2):
        k, v = _contig(x.k_pool, x, b), _contig(x.v_pool, x, b)
        for h in range(2):
            sc = k[h] @ x.q[b, h].double()
            top2 = torch.topk(sc, 2).values
            assert (top2[0] - top2[1]) * big > 60  # limit reached in fp64
            want = v[h, int(torch.argmax(sc))].numpy()
            if not np.allclose(out[b, h], want, rtol=0, atol=1e-12):
                return False
    return True


def _bf16(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def _pin_int8_codes(lib):
    # round half to even on x / scale, clamped to +-127; NaN -> 0
    x = _bf16([1.0, 0.25, 0.75, 1.25, -0.75, 100.0, -100.0, float("nan"),
               float("inf"), float("-inf"), 2.5, -1.25, 0.0, 63.75, -63.75])
    want = [2, 0, 2, 2, -2, 127, -127, 0, 127, -127, 5, -2, 0, 127, -127]
    codes, st = oracle.quantize_int8(x, 0.5, lib=lib, return_status=True)
    if st != oracle.OK or codes.tolist() != want:
        return False
    # exact multiples of a power-of-two scale come back as themselves
    c = np.arange(-127, 128)
    codes = oracle.quantize_int8(_bf16((c / 64.0).tolist()), 1.0 / 64, lib=lib)
    if codes.tolist() != c.tolist():
        return False
    bad, st = oracle.quantize_int8(x, 0.0, lib=lib, return_status=True)
    return st == oracle.ERR_SCALE and not bad.any()


def _pin_int8_write(lib):
    nb, bs, hkv, d = 4, 8, 2, 2
    kp = np.zeros((nb, bs, hkv, d), np.int8)
    vp = np.zeros((nb, bs, hkv, d), np.int8)
    kn = _bf16([[[1.0, -2.0], [3.0, 4.0]]])
    vn = _bf16([[[0.5, 0.25], [-1.0, 8.0]]])
    st = oracle.write_int8(kp, vp, kn, vn, np.array([2 * bs + 3]), bs,
                           [0.5, 1.0], [0.25, 2.0], lib=lib)
    return (st == oracle.OK and kp[2, 3].tolist() == [[2, -4], [3, 4]]
            and vp[2, 3].tolist() == [[2, 1], [0, 4]]
            and int(np.abs(kp).sum()) == 13 and int(np.abs(vp).sum()) == 7)


def _pin_int8_decode(lib):
    # INT8 pools whose dequantised values are exact in bf16 must decode
    # exactly like bf16 pools holding those values (the pinned 16-bit path)
    x = W.make_inputs(_cfg("decode", 4, 2, 64, 16, 24, [1, 37, 90], "identity",
                           dtype="bf16"), seed=47)
    rng = np.random.default_rng(5)
    shape = tuple(x.k_pool.shape)
    kc = rng.integers(-127, 128, shape).astype(np.int8)
    vc = rng.integers(-127, 128, shape).astype(np.int8)
    ks, vs = np.array([2.0 ** -6, 2.0 ** -4], np.float32), np.array([2.0 ** -3, 2.0 ** -7], np.float32)
    kb = torch.from_numpy(kc.astype(np.float32) * ks[None, None, :, None]).to(torch.bfloat16)
    vb = torch.from_numpy(vc.astype(np.float32) * vs[None, None, :, None]).to(torch.bfloat16)
    want = oracle.decode(x.q, kb, vb, x.block_table, x.context_lens, 2, 16, x.scale,
                         lib=lib)
    got = oracle.decode_int8(x.q, kc, vc, x.block_table, x.context_lens, 2, 16, x.scale,
                             ks, vs, lib=lib)
    return np.array_equal(got, want)


def _pin_int8_nearest(lib):
    # every code is the nearest integer to x / scale (ties to even), clamped
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 3).to(torch.bfloat16)
    s = np.float32(0.0371)
    y = x.float().numpy() / s
    c = oracle.quantize_int8(x, float(s), lib=lib).astype(np.float64)
    inside = np.abs(y) < 127
    ci = c[inside]
    err = np.abs(y[inside] - ci)
    ties = err == 0.5
    return (bool((err <= 0.5).all()) and bool((ci[ties] % 2 == 0).all())
            and bool((c[~inside] == np.sign(y[~inside]) * 127).all()))


def _pin_copy_blocks(lib):
    # block dst of both pools becomes block src byte for byte, pair by pair;
    # a pair naming a block outside the pool copies nothing and is reported
    rng = np.random.default_rng(12)
    shape = (7, 4, 2, 8)

    def check(k0, v0, pairs, status, moved):
        k, v = k0.copy(), v0.copy()
        st = oracle.copy_blocks(k, v, pairs, lib=lib)
        wk, wv = k0.copy(), v0.copy()
        for src, dst in moved:
            wk[dst], wv[dst] = k0[src], v0[src]
        return st == status and np.array_equal(k, wk) and np.array_equal(v, wv)

    k16 = rng.integers(0, 1 << 16, shape, dtype=np.uint16)
    v16 = rng.integers(0, 1 << 16, shape, dtype=np.uint16)
    k8 = rng.integers(-128, 128, shape, dtype=np.int8)
    v8 = rng.integers(-128, 128, shape, dtype=np.int8)
    return (check(k16, v16, [[1, 4], [3, 0], [5, 5]], oracle.OK, [(1, 4), (3, 0)])
            and check(k16, v16, [[7, 2], [2, -1], [6, 1]], oracle.ERR_BLOCK, [(6, 1)])
            and check(k8, v8, [[0, 6]], oracle.OK, [(0, 6)])
            and check(k8, v8, [], oracle.OK, []))


def _pin_copy_on_write_decode(lib):
    # [ATB] copy-on-write: B forks from A and shares A's blocks; before it
    # appends its own token it copies the shared, partly filled last block
    # to a free block.  B then attends to A's tokens plus its own, and A
    # still to its own only -- as if each sequence sat alone, contiguously.
    # (The pool and block-table rows are roomier than needed so that every
    # planted mistake -- e.g. a write offset of slot / bs -- stays in bounds.)
    rng = np.random.default_rng(21)
    bs, hkv, hq, d, nb = 4, 2, 4, 8, 16
    L = 2 * bs + 3

    def f16(shape):
        return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.float16)

    def u16(t):
        return t.view(torch.int16).numpy().view(np.uint16)
    ka, va, kb, vb = f16((L, hkv, d)), f16((L, hkv, d)), f16((1, hkv, d)), f16((1, hkv, d))
    kp = np.zeros((nb, bs, hkv, d), np.uint16)
    vp = np.zeros_like(kp)
    a_blocks = [5, 2, 7]
    oracle.write(kp, vp, ka, va, np.array([a_blocks[j // bs] * bs + j % bs for j in range(L)]),
                 bs, lib=lib)
    st = oracle.copy_blocks(kp, vp, [[7, 0]], lib=lib)
    oracle.write(kp, vp, kb, vb, np.array([0 * bs + L % bs]), bs, lib=lib)
    q = f16((2, hq, d))
    lens = np.array([L, L + 1], np.int32)
    got = oracle.decode(q, kp, vp, np.array([[5, 2, 7, -1], [5, 2, 0, -1]], np.int32), lens,
                        hkv, bs, 0.3, lib=lib)
    kr = np.zeros((6, bs, hkv, d), np.uint16)
    vr = np.zeros_like(kr)
    for base in (0, 3 * bs):
        kr.reshape(-1, hkv, d)[base:base + L] = u16(ka)
        vr.reshape(-1, hkv, d)[base:base + L] = u16(va)
    kr.reshape(-1, hkv, d)[3 * bs + L] = u16(kb)[0]
    vr.reshape(-1, hkv, d)[3 * bs + L] = u16(vb)[0]
    want = oracle.decode(q, kr, vr, np.array([[0, 1, 2, -1], [3, 4, 5, -1]], np.int32), lens,
                         hkv, bs, 0.3, lib=lib)
    return st == oracle.OK and np.array_equal(got, want)


def _pin_fp8_codes(lib):
    # the E4M3 table against torch's float8_e4m3fn (a library routine) and
    # closed forms; the encoder against torch's round-to-nearest-even inside
    # the range, ties to the even code, saturation at 448, NaN -> 0, -0 kept
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.fp8_value(codes, lib=lib)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(t)
    if not (np.array_equal(np.isnan(v), nan) and np.array_equal(v[~nan], t[~nan])):
        return False
    if not (v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6
            and v[0x38] == 1.0 and v[0xB8] == -1.0):
        return False
    rng = np.random.default_rng(13)
    for s in (1.0, 0.01, 37.0):
        x = torch.from_numpy(rng.standard_normal(4096).astype(np.float32) * 40).to(torch.bfloat16)
        y = x.float() / np.float32(s)
        inside = (y.abs() < 448).numpy()
        c = oracle.quantize_fp8(x, s, lib=lib)
        want = y[torch.from_numpy(inside)].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        if not np.array_equal(c[inside], want):
            return False
        if not (c[~inside] & 0x7F == 0x7E).all():
            return False
    ties = _bf16([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, -1.0625, 500.0, -1e4,
                  float("nan"), -0.0, float("inf")])
    c, st = oracle.quantize_fp8(ties, 1.0, lib=lib, return_status=True)
    if st != oracle.OK or c.tolist() != [0x38, 0x3A, 0x00, 0x02, 0xB8, 0x7E, 0xFE, 0x00, 0x80,
                                         0x7E]:
        return False
    bad, st = oracle.quantize_fp8(ties, -1.0, lib=lib, return_status=True)
    return st == oracle.ERR_SCALE and not bad.any()


def _pin_fp8_write(lib):
    # code = sign << 7 | exponent field << 3 | fraction, worked by hand
    nb, bs, hkv, d = 4, 8, 2, 2
    kp = np.zeros((nb, bs, hkv, d), np.uint8)
    vp = np.zeros((nb, bs, hkv, d), np.uint8)
    kn = _bf16([[[1.0, -2.0], [3.0, 4.0]]])   # / [0.5, 1.0] -> 2, -4 | 3, 4
    vn = _bf16([[[0.5, 0.25], [-1.0, 8.0]]])  # / [0.25, 2.0] -> 2, 1 | -0.5, 4
    st = oracle.write_fp8(kp, vp, kn, vn, np.array([2 * bs + 3]), bs, [0.5, 1.0],
                          [0.25, 2.0], lib=lib)
    return (st == oracle.OK and kp[2, 3].tolist() == [[0x40, 0xC8], [0x44, 0x48]]
            and vp[2, 3].tolist() == [[0x40, 0x38], [0xB0, 0x48]]
            and int(kp.astype(np.int64).sum()) == 0x40 + 0xC8 + 0x44 + 0x48)


def _pin_fp8_decode(lib):
    # FP8 pools whose dequantised values are exact in bf16 decode exactly
    # like bf16 pools holding those values (the pinned 16-bit path)
    x = W.make_inputs(_cfg("decode", 4, 2, 64, 16, 24, [1, 37, 90], "identity",
                           dtype="bf16"), seed=48)
    rng = np.random.default_rng(6)
    shape = tuple(x.k_pool.shape)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    kc, vc = rng.choice(finite, shape), rng.choice(finite, shape)
    ks = np.array([2.0 ** -3, 2.0 ** 2], np.float32)
    vs = np.array([2.0 ** 1, 2.0 ** -5], np.float32)
    kv = oracle.fp8_value(kc, lib=lib) * ks[None, None, :, None]
    vv = oracle.fp8_value(vc, lib=lib) * vs[None, None, :, None]
    kb = torch.from_numpy(kv).to(torch.bfloat16)
    vb = torch.from_numpy(vv).to(torch.bfloat16)
    if not (np.array_equal(kb.double().numpy(), kv) and np.array_equal(vb.double().numpy(), vv)):
        return False
    want = oracle.decode(x.q, kb, vb, x.block_table, x.context_lens, 2, 16, x.scale, lib=lib)
    got = oracle.decode_fp8(x.q, kc, vc, x.block_table, x.context_lens, 2, 16, x.scale,
                            ks, vs, lib=lib)
    return np.array_equal(got, want)


PINS = [_pin_decode_sdpa, _pin_prefill_sdpa, _pin_chunked_tail,
        _pin_decoders, _pin_write, _pin_saturated_softmax, _pin_int8_codes,
        _pin_int8_write, _pin_int8_decode, _pin_int8_nearest, _pin_copy_blocks,
        _pin_copy_on_write_decode, _pin_fp8_codes, _pin_fp8_write, _pin_fp8_decode]


@pytest.fixture(scope="module")
def tmpdir_mod():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmodified_oracle_passes_every_pin(tmpdir_mod):
    lib = _build(tmpdir_mod, "clean", None)
    assert all(p(lib) for p in PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmpdir_mod, name):
    lib = _build(tmpdir_mod, name, MUTANTS[name])
    failed = [p.__name__ for p in PINS if not p(lib)]
    assert failed, f"mutant {name} passed every pin"
