"""Parity at the edges of the supported sizes, against the oracle.

- Caches larger than 2 GiB: block ids whose byte offsets pass 2^31 and 2^32
  (64-bit address arithmetic in every gather, in the new-token write and in
  the TMA coordinates), a 65,536-token context split 64 ways and merged.
- The ragged-balanced plan at its largest batch (2,048 sequences) and one
  sequence past it (the per-partition plan takes over).
- Scatter of 100,000 tokens and copy of 4,000 block pairs, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, max_err, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def assert_clean_status():
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0


def test_decode_append_over_4gib_caches():
    """Two sequences (65,536 and 1,000 tokens) whose blocks all sit past the
    first 2 GiB of a 4 GiB-per-cache pool; the new tokens land there too."""
    nb, bs, hkv, d, hq = 1 << 17, 16, 8, 128, 32          # 131,072 blocks x 32 KiB = 4 GiB per cache
    lens = np.array([65536, 1000], np.int32)
    need = [workloads.cdiv(int(n), bs) for n in lens]
    rng = np.random.default_rng(1717)
    ids = rng.permutation(np.arange(nb // 2 + 1000, nb, dtype=np.int32))[:sum(need)]
    assert int(ids.min()) * bs * hkv * d * 2 >= 2 ** 31
    tables = np.zeros((2, max(need)), np.int32)
    tables[0, :need[0]] = ids[:need[0]]
    tables[1, :need[1]] = ids[need[0]:]
    used = ids
    shape_blk = (used.size, bs, hkv, d)
    k_used = workloads.bf16_round(rng.standard_normal(shape_blk, dtype=np.float32))
    v_used = workloads.bf16_round(rng.standard_normal(shape_blk, dtype=np.float32))
    query = workloads.bf16_round(rng.standard_normal((2, hq, d), dtype=np.float32))
    new_k = workloads.bf16_round(rng.standard_normal((2, hkv, d), dtype=np.float32))
    new_v = workloads.bf16_round(rng.standard_normal((2, hkv, d), dtype=np.float32))
    scale = 1.0 / np.sqrt(d)

    k_cache = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros_like(k_cache)
    idx = torch.from_numpy(used.astype(np.int64)).cuda()
    k_cache.index_copy_(0, idx, to_dev(k_used))
    v_cache.index_copy_(0, idx, to_dev(v_used))
    out = torch.full((2, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    mcl = int(lens.max())
    n = pa.pa_decode_workspace_size(2, hq, hkv, d, bs, mcl)
    ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
    plan = pa.pa_decode_plan(2, hq, hkv, d, bs, mcl, with_workspace=True)
    assert plan["num_splits"] > 8 and not plan["cluster_merge"], plan
    pa.pa_decode_append(out, to_dev(query), to_dev(new_k), to_dev(new_v), k_cache, v_cache, to_dev(tables),
                        to_dev(lens), mcl, scale, workspace=ws)
    torch.cuda.synchronize()

    # oracle over a compact pool holding just the used blocks (same values, renumbered)
    remap = np.zeros(nb, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    ctables = remap[tables]
    ck, cv = k_used.copy(), v_used.copy()
    slots = oracle.slot_mapping(ctables, np.arange(2), lens - 1, bs)
    oracle.reshape_and_cache(ck, cv, new_k, new_v, slots)
    want = oracle.paged_attention(query, ck, cv, ctables, lens, scale)
    assert max_err(out, want) <= ATOL
    # the blocks holding the new tokens, read back: bit for bit
    for b in range(2):
        blk = int(tables[b, (lens[b] - 1) // bs])
        got_k = to_host_bits(k_cache[blk])
        got_v = to_host_bits(v_cache[blk])
        assert np.array_equal(got_k, ck[remap[blk]]) and np.array_equal(got_v, cv[remap[blk]])
    assert_clean_status()


@pytest.mark.parametrize("num_seqs", [2048, 2049])
def test_balanced_plan_at_its_batch_limit(num_seqs):
    rng = np.random.default_rng(num_seqs)
    lens = rng.integers(1, 300, size=num_seqs).astype(np.int32)
    hq, hkv, d, bs = 8, 2, 128, 16
    need = sum(workloads.cdiv(int(x), bs) for x in lens)
    batch = workloads.make_batch("limit", lens, hq, hkv, d, bs, need + 17, True, seed_values=num_seqs + 1)
    plan = pa.pa_decode_plan(num_seqs, hq, hkv, d, bs, int(lens.max()), with_workspace=True)
    assert plan["balanced"] == (1 if num_seqs <= 2048 else 0), plan
    db = DeviceBatch(batch)
    ws = make_workspace(batch)
    out = torch.full((num_seqs, hq, d), float("nan"), dtype=torch.float32, device="cuda")
    pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, batch.max_context_len, batch.scale, workspace=ws)
    torch.cuda.synchronize()
    k, v = batch.k_cache.copy(), batch.v_cache.copy()
    slots = oracle.slot_mapping(batch.block_tables, np.arange(num_seqs), lens - 1, bs)
    oracle.reshape_and_cache(k, v, batch.new_key, batch.new_value, slots)
    want = oracle.paged_attention(batch.query, k, v, batch.block_tables, lens, batch.scale)
    assert max_err(out, want) <= ATOL
    assert np.array_equal(to_host_bits(db.k_cache), k) and np.array_equal(to_host_bits(db.v_cache), v)
    assert_clean_status()


def test_scatter_and_copy_at_scale():
    rng = np.random.default_rng(4242)
    nb, bs, hkv, d = 8192, 16, 8, 128
    k = rng.integers(0, 2 ** 16, size=(nb, bs, hkv, d)).astype(np.uint16)
    v = rng.integers(0, 2 ** 16, size=(nb, bs, hkv, d)).astype(np.uint16)
    kd, vd = to_dev(k), to_dev(v)
    # 100,000 tokens into distinct slots of the 131,072
    T = 100_000
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    key = rng.integers(0, 2 ** 16, size=(T, hkv, d)).astype(np.uint16)
    val = rng.integers(0, 2 ** 16, size=(T, hkv, d)).astype(np.uint16)
    pa.pa_reshape_and_cache(to_dev(key), to_dev(val), kd, vd, torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache(k, v, key, val, slots)
    # 4,000 copy-on-write pairs: distinct destinations, disjoint from the sources
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:4000], perm[4000:8000]], axis=1).astype(np.int64)
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(k, v, pairs)
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert_clean_status()
