"""Pins for the oracle's index handling: the pages' printed worked examples
(tests/golden/index_examples.json), exact 16-bit decoding, and the cache
write's bit-copy semantics.  CPU only."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_34_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "index_examples.json")))


@pytest.mark.parametrize("ex", GOLDEN["slot_of"], ids=lambda e: str(e["slot"]))
def test_slot_of_worked_example(ex):
    bs = ex["block_size"]
    e = ex["block_table_entry"]
    table = np.full((e["row"] + 1, e["col"] + 1), -1, dtype=np.int32)
    table[e["row"], e["col"]] = e["value"]
    assert ex["seq_pos"] // bs == ex["logical_block"]
    assert ex["seq_pos"] % bs == ex["offset"]
    assert oracle.slot_of(table, ex["batch_idx"], ex["seq_pos"], bs) == ex["slot"]


@pytest.mark.parametrize("ex", GOLDEN["static_block_table"], ids=lambda e: "bt")
def test_static_block_table(ex):
    t = oracle.static_block_table(ex["batch_size"], ex["max_seq_len"], ex["block_size"])
    assert t == ex["table"]
    assert len(t[0]) == ex["blocks_per_seq"]
    assert sum(len(r) for r in t) == ex["total_blocks"]


@pytest.mark.parametrize("ex", GOLDEN["prefill_slots"], ids=lambda e: "prefill")
def test_prefill_slots(ex):
    got = oracle.sequential_prefill_slots(ex["kv_len"], ex["max_seq_len"])
    want = []
    for lo, hi in ex["ranges"]:
        want.extend(range(lo, hi + 1))
    assert got == want and len(got) == ex["length"]


@pytest.mark.parametrize("ex", GOLDEN["decode_slots"], ids=lambda e: "decode")
def test_decode_slots(ex):
    assert oracle.sequential_decode_slots(ex["kv_len"], ex["max_seq_len"]) == \
        ex["slot_mapping"]
    # The sequential pool is the static block table: the same slots follow
    # from the general mapping through that table (the pages' "the two
    # address the same way").
    bs = 128
    table = oracle.static_block_table(len(ex["kv_len"]), ex["max_seq_len"], bs)
    for b, n in enumerate(ex["kv_len"]):
        assert oracle.slot_of(table, b, n, bs) == ex["slot_mapping"][b][0]


@pytest.mark.parametrize("ex", GOLDEN["actual_seq_lengths"], ids=lambda e: str(e["tnd"]))
def test_actual_seq_lengths(ex):
    assert oracle.tnd_actual_seq_lengths(ex["lengths"]) == ex["tnd"]


@pytest.mark.parametrize("ex", GOLDEN["cu_seqlens"], ids=lambda e: str(e["cu_seqlens"]))
def test_cu_seqlens(ex):
    cu = oracle.cu_seqlens(ex["lengths"])
    assert cu == ex["cu_seqlens"]
    assert len(cu) == len(ex["lengths"]) + 1 and cu[0] == 0
    if "total_tokens" in ex:
        assert cu[-1] == ex["total_tokens"]
        assert max(ex["lengths"]) == ex["max_seq_len_in_batch"]


@pytest.mark.parametrize("ex", GOLDEN["blocks_needed"], ids=lambda e: str(e["blocks"]))
def test_blocks_needed(ex):
    assert oracle.blocks_needed(ex["num_tokens"], ex["block_size"]) == ex["blocks"]


def test_f16_decoder_exhaustive():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode16(pats, oracle.F16)
    want = pats.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, want)  # NaNs compare equal here


def test_bf16_decoder_exhaustive():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode16(pats, oracle.BF16)
    want = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(got, want)


def _pool(nb, bs, hkv, d, fill=0x7E00):
    return np.full((nb, bs, hkv, d), fill, dtype=np.uint16)


def test_write_is_bit_copy_and_leaves_other_rows():
    rng = np.random.default_rng(1)
    nb, bs, hkv, d = 6, 4, 3, 8
    kp, vp = _pool(nb, bs, hkv, d), _pool(nb, bs, hkv, d)
    n = 7
    kn = rng.integers(0, 65536, size=(n, hkv, d)).astype(np.uint16)
    vn = rng.integers(0, 65536, size=(n, hkv, d)).astype(np.uint16)
    slots = np.array([5, -1, 0, 23, 9, -7, 12], dtype=np.int64)
    assert oracle.write(kp, vp, kn, vn, slots, bs) == oracle.OK
    flat_k, flat_v = kp.reshape(nb * bs, hkv, d), vp.reshape(nb * bs, hkv, d)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(flat_k[s], kn[t])
        np.testing.assert_array_equal(flat_v[s], vn[t])
        written.add(int(s))
    for r in range(nb * bs):
        if r not in written:
            assert (flat_k[r] == 0x7E00).all() and (flat_v[r] == 0x7E00).all()


def test_write_block_and_offset_split():
    # slot s lands in block s // bs at offset s % bs: check through the 4-D
    # index, not the flat view.
    nb, bs, hkv, d = 5, 8, 1, 2
    kp, vp = _pool(nb, bs, hkv, d, 0), _pool(nb, bs, hkv, d, 0)
    kn = np.array([[[111, 222]]], dtype=np.uint16)
    assert oracle.write(kp, vp, kn, kn, np.array([3 * bs + 5]), bs) == oracle.OK
    assert (kp[3, 5, 0] == [111, 222]).all()
    assert kp.sum() == 333


def test_write_out_of_range_slot_reported_and_skipped():
    nb, bs, hkv, d = 2, 4, 1, 4
    kp, vp = _pool(nb, bs, hkv, d, 0), _pool(nb, bs, hkv, d, 0)
    kn = np.ones((2, hkv, d), dtype=np.uint16)
    st = oracle.write(kp, vp, kn, kn, np.array([nb * bs, 1]), bs)
    assert st == oracle.ERR_SLOT
    assert kp.reshape(-1, d)[1].tolist() == [1, 1, 1, 1]
    assert kp.sum() == 4


@pytest.mark.parametrize("name", W.ORDER)
def test_generator_placement_matches_slot_formula(name):
    # The generator lays out the pool (allocator role).  Its slot_mapping
    # must agree with the pages' mapping formula applied to its block table,
    # and its block tables must never share a block between sequences.
    lengths = None
    if name == "long-context-decode":
        lengths = [40000, 33000, 1000, 5000]
    x = W.make_inputs(name, lengths=lengths, write_new_token=True) \
        if W.CONFIGS[name]["kind"] == "decode" else W.make_inputs(name)
    bt = x.block_table.numpy()
    ctx = x.context_lens.numpy()
    nl = x.new_lens.numpy()
    slots = x.slot_mapping.numpy()
    k = 0
    for b in range(x.num_seqs):
        for pos in range(ctx[b] - nl[b], ctx[b]):
            assert slots[k] == oracle.slot_of(bt, b, pos, x.block_size)
            k += 1
    assert k == len(slots)
    used = bt[bt >= 0]
    assert len(np.unique(used)) == len(used)
    assert used.max(initial=0) < x.num_blocks
    for b in range(x.num_seqs):
        assert (bt[b, :oracle.blocks_needed(ctx[b], x.block_size)] >= 0).all()
