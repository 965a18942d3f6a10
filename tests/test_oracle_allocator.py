"""Pins for the oracle's block-manager model, slot formula, scatter and copy,
against the worked numbers the pages print (tests/golden/pages_numbers.json)."""
import math

import numpy as np
import pytest

import oracle
from oracle import BlockManagerModel, OutOfBlocks
import workloads


def cdiv(a, b):
    return -(-a // b)


def test_toy_three_requests(golden):
    g = golden["toy_three_requests"]
    B = g["block_size"]
    order = [3, 7, 0, 5, 9, 4] + [b for b in range(g["pool_blocks"]) if b not in (3, 7, 0, 5, 9, 4)]
    bm = BlockManagerModel(g["pool_blocks"], B, reserve_null_block=False, free_order=order)
    for seq, n in enumerate(g["lens"]):
        bm.allocate(seq, n)
    assert [len(bm.block_table(s)) for s in range(3)] == g["blocks"]
    assert [bm.block_table(s) for s in range(3)] == g["tables"]
    st = bm.stats()
    assert st["logical_blocks"] * B == g["paged_slots"]
    assert st["num_tokens"] == g["tokens"]
    assert st["waste_slots"] == g["waste_slots"]
    assert [len(bm.block_table(s)) * B - n for s, n in enumerate(g["lens"])] == g["padding_slots"]
    assert st["free_blocks"] == g["free_blocks_after"]
    assert len(g["lens"]) * g["contiguous_budget"] == g["contiguous_slots"]
    assert g["contiguous_slots"] // g["paged_slots"] == g["ratio"]
    # request B grows: its 48th token still fits block 9, the 49th takes block 11
    bm.free = [11] + [b for b in bm.free if b != 11]
    bm.append_slot(1)
    assert bm.block_table(1) == g["tables"][1]
    bm.append_slot(1)
    assert bm.block_table(1) == g["b_table_after_growth"]
    # the page's "+20 tokens" would need cdiv(67, 16) = 5 blocks, not 4
    for _ in range(20 - 2):
        bm.append_slot(1)
    assert bm.num_tokens(1) == 67 and len(bm.block_table(1)) == cdiv(67, 16) == 5


def test_block_size_tradeoff(golden):
    g = golden["block_size_tradeoff_47_tokens"]
    for row in g["rows"]:
        bm = BlockManagerModel(64, row["block_size"], reserve_null_block=False)
        bm.allocate(0, g["tokens"])
        assert len(bm.block_table(0)) == row["lookups"]
        assert bm.stats()["waste_slots"] == row["wasted"]


def test_incremental_fill(golden):
    g = golden["incremental_fill"]
    B = g["block_size"]
    bm = BlockManagerModel(32, B, reserve_null_block=False, free_order=g["free_list"])
    bm.allocate(0, g["prompt_tokens"])
    assert bm.block_table(0) == g["table_after_prefill"]
    for pos in (6, 7, 8):
        slot, src, dst = bm.append_slot(0)
        assert (src, dst) == (-1, -1)
        assert slot // B == g["slot_block_of_position"][str(pos)]
        assert slot % B == pos % B
    assert bm.block_table(0) == g["table_after_third_block"]
    bm.free_seq(0)
    assert bm.free[:3] == g["returned_on_finish"]
    assert sorted(bm.free) == sorted(g["free_list"])


def test_cdiv_examples(golden):
    g = golden["cdiv_examples"]
    for row in g["rows"]:
        bm = BlockManagerModel(64, row["block_size"], reserve_null_block=False)
        bm.allocate(0, row["tokens"])
        assert len(bm.block_table(0)) == row["blocks"]
        if "wasted" in row:
            assert bm.stats()["waste_slots"] == row["wasted"]
        if "slots" in row:
            assert bm.stats()["logical_blocks"] * row["block_size"] == row["slots"]
    h = g["hundred_requests"]
    bm = BlockManagerModel(100 * 19 + 1, 16)
    for s in range(100):
        bm.allocate(s, h["avg_tokens"])
    st = bm.stats()
    assert st["logical_blocks"] * 16 == h["paged_units"]
    assert st["num_tokens"] == h["used_units"]
    assert 100 * h["max_tokens"] == h["static_units"]
    # waste is under one block per request ("PagedAttention, explained.", waste bound)
    assert st["waste_slots"] < 100 * 16


def test_slot_formula(golden):
    g = golden["slot_of_token_53"]
    table = np.array([[40, 41, 42, 77, 43]], np.int32)
    slot = oracle.slot_mapping(table, [0], [g["position"]], g["block_size"])[0]
    assert slot // g["block_size"] == table[0, g["logical_block"]]
    assert slot % g["block_size"] == g["offset"]
    assert oracle.slot_mapping(table, [0], [-1], 16)[0] == -1


def test_cow_clone(golden):
    g = golden["cow_clone"]
    bm = BlockManagerModel(8, 16, reserve_null_block=False)
    bm.allocate(0, 20)                 # A: system prompt spills into P1
    bm.fork(0, 1)                      # B shares P0, P1
    assert bm.block_table(1) == g["shared_tables"]
    assert bm.refcount[0] == bm.refcount[1] == 2
    slot, src, dst = bm.append_slot(1)  # B writes into the shared P1
    assert [src, dst] == g["pair"]
    assert bm.block_table(1) == g["writer_table_after"]
    assert bm.block_table(0) == g["other_table_after"]
    assert bm.refcount[1] == 1 and bm.refcount[2] == 1 and bm.refcount[0] == 2
    assert slot == 2 * 16 + 20 % 16
    # A now writes in place: its count is back to one
    slot, src, dst = bm.append_slot(0)
    assert (src, dst) == (-1, -1) and slot == 1 * 16 + 20 % 16


def test_null_block_never_handed_out():
    bm = BlockManagerModel(5, 4)
    bm.allocate(0, 16)
    assert 0 not in bm.block_table(0)
    with pytest.raises(OutOfBlocks):
        bm.allocate(1, 1)
    assert bm.stats()["free_blocks"] == 0


def test_qwen3_capacity(golden):
    g = golden["qwen3_8b_capacity"]
    per_token = g["layers"] * g["kv_heads"] * g["head_dim"] * 2 * g["bytes_per_value"]
    assert per_token == g["bytes_per_token"] == 144 * 1024
    assert g["cache_tokens"] // g["block_size"] == g["blocks"] == workloads.QWEN3_POOL_BLOCKS
    assert round(g["cache_tokens"] / g["max_len"], 2) == g["max_concurrency"]
    assert g["request_tokens"] == workloads.QWEN3_TOKENS
    # no sharing: 16 x 261 blocks
    bm = BlockManagerModel(g["blocks"] + 1, g["block_size"])
    for s in range(g["in_flight"]):
        bm.allocate(s, g["request_tokens"])
        assert len(bm.block_table(s)) == g["blocks_per_request"]
    used = bm.stats()["used_blocks"]
    assert round(100 * used / g["blocks"], 1) == g["usage_percent_no_sharing"]
    # one shared 4,000-token prefix: 250 shared blocks + 11 private per request
    bm = BlockManagerModel(g["blocks"] + 1, g["block_size"])
    bm.allocate(0, g["prefix_tokens"])
    for s in range(1, g["in_flight"]):
        bm.fork(0, s)
    for s in range(g["in_flight"]):
        for _ in range(g["private_tokens"]):
            _, src, dst = bm.append_slot(s)
            assert src == -1
    st = bm.stats()
    assert st["shared_blocks"] == g["shared_prefix_blocks"]
    assert st["used_blocks"] == g["blocks_with_sharing"]
    assert len(bm.block_table(0)) - g["shared_prefix_blocks"] == g["private_blocks_per_request"]
    assert round(100 * st["used_blocks"] / g["blocks"], 1) == g["usage_percent_with_sharing"]


def test_opt13b_kv(golden):
    g = golden["opt13b_kv"]
    per_token = 2 * g["hidden"] * g["layers"] * g["bytes_per_value"]
    assert per_token == g["bytes_per_token"]
    assert round(per_token * g["tokens"] / 2**30, 1) == g["gigabytes"]


def test_shared_prefix_cow_counts():
    """Prefix of 2,064 tokens at block size 32: 64 full blocks plus one half-full
    shared block. Under the refcount rule the first 63 writers clone it and the
    last finds its count at one and writes in place."""
    S = 64
    bm = BlockManagerModel(4096, 32)
    bm.allocate(0, 2064)
    for s in range(1, S):
        bm.fork(0, s)
    pairs = []
    for s in range(S):
        _, src, dst = bm.append_slot(s)
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == S - 1
    assert len({d for _, d in pairs}) == S - 1
    assert {s for s, _ in pairs} == {bm.block_table(S - 1)[64]}
    # the literal 2,048-token prefix is 64 full blocks: no copy at all
    bm = BlockManagerModel(4096, 32)
    bm.allocate(0, 2048)
    for s in range(1, S):
        bm.fork(0, s)
    assert all(bm.append_slot(s)[1] == -1 for s in range(S))
    assert bm.stats()["shared_blocks"] == 64


def test_scatter_and_copy():
    rng = np.random.default_rng(0)
    nb, B, hkv, d = 6, 4, 2, 8
    k = rng.standard_normal((nb, B, hkv, d)).astype(np.float32)
    v = rng.standard_normal((nb, B, hkv, d)).astype(np.float32)
    k0, v0 = k.copy(), v.copy()
    key = rng.standard_normal((3, hkv, d)).astype(np.float32)
    val = rng.standard_normal((3, hkv, d)).astype(np.float32)
    slots = [5, -1, 22]
    oracle.reshape_and_cache(k, v, key, val, slots)
    flat_k, flat_v = k.reshape(nb * B, hkv, d), v.reshape(nb * B, hkv, d)
    assert np.array_equal(flat_k[5], key[0]) and np.array_equal(flat_v[22], val[2])
    changed = np.any(k.reshape(nb * B, -1) != k0.reshape(nb * B, -1), axis=1)
    assert set(np.nonzero(changed)[0]) == {5, 22}
    k1, v1 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, [(1, 4), (2, 0)])
    assert np.array_equal(k[4], k1[1]) and np.array_equal(v[0], v1[2])
    for b in (1, 2, 3, 5):
        assert np.array_equal(k[b], k1[b]) and np.array_equal(v[b], v1[b])
