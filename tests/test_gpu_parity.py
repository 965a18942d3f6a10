"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Scatter and block copy must be bit-exact; attention must stay within 2e-3
max abs error (bf16 K/V, fp32 accumulation; "What Does PagedAttention
Actually Optimize?", section 8: paging does not change the result)."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import (ATOL, DeviceBatch, make_workspace, max_err, new_token_slots, oracle_step,
                       run_step, to_dev, to_host_bits)

pytestmark = pytest.mark.gpu


def assert_clean_status():
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0


# ---------------------------------------------------------------------------
# small shapes: several tiles, ragged tails, every kernel variant
# ---------------------------------------------------------------------------
SMALL = [
    # lens, Hq, Hkv, D, block_size, bf16
    ((25, 47, 12), 4, 4, 64, 16, False),           # the pages' toy (fp32: CUDA-core kernel)
    ((1, 2, 15, 16, 17, 100, 333), 8, 2, 128, 16, True),
    ((1, 7, 8, 9, 64, 250), 16, 4, 128, 8, True),
    ((1, 31, 32, 33, 700), 32, 8, 128, 32, True),
    ((5, 40, 129), 4, 4, 64, 16, True),            # G = 1
    ((3, 77, 300), 16, 1, 64, 32, True),           # G = 16, one full tile of heads
    ((50, 260), 64, 2, 128, 16, True),             # G = 32: two head tiles
    ((19, 90), 8, 2, 128, 4, True),                # blocks of 4: rows gathered by 16-byte copies
    ((1, 3, 16, 17, 95, 400), 16, 4, 128, 1, True),  # blocks of 1: 16 table entries per tile
    ((2, 33, 64, 250), 8, 8, 64, 2, True),         # blocks of 2, G = 1
    ((9, 700), 24, 12, 128, 4, True),              # blocks of 4, groups of 6 heads, split
    ((7, 130), 4, 1, 64, 4, True),                 # one KV head: 8 chunks per token row
    ((12, 40), 8, 2, 128, 12, True),               # block size not a power of two: CUDA-core kernel
    ((19, 90), 8, 2, 64, 64, True),
    ((10, 45), 6, 3, 64, 16, False),
    ((33, 200, 17), 24, 12, 128, 16, True),        # 12 KV heads: groups of 6 per CTA
    ((70, 300), 32, 16, 64, 32, True),             # 16 KV heads: two groups of 8
    ((5, 600), 12, 3, 128, 128, True),             # large blocks: 8 tiles per block
    ((5, 700), 8, 2, 128, 256, True),              # the largest blocks: tiles at offsets up to 240
    ((3, 513), 64, 1, 64, 256, True),              # G = 64: four head tiles over one KV head
]


@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("use_ws", [False, True])
def test_decode_small(case, use_ws):
    lens, Hq, Hkv, D, bs, bf16 = SMALL[case]
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("small", lens, Hq, Hkv, D, bs, need + 13, bf16,
                                 seed_values=500 + case, seed_blocks=600 + case)
    db = DeviceBatch(batch)
    ws = make_workspace(batch) if use_ws else None
    out = run_step(db, workspace=ws)
    want, k_want, v_want = oracle_step(batch)
    assert np.array_equal(to_host_bits(db.k_cache), k_want)
    assert np.array_equal(to_host_bits(db.v_cache), v_want)
    err = max_err(out, want)
    assert err <= ATOL, err
    if use_ws:   # the workspace is reusable as left: a second call gives the same answer
        out2 = torch.empty_like(out)
        pa.pa_decode(out2, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                     batch.max_context_len, batch.scale, workspace=ws)
        assert torch.equal(out, out2)
    assert_clean_status()


@pytest.mark.parametrize("bs", [16, 8, 4, 1])
def test_decode_nan_in_unused_slots_and_table_tail(bs):
    """Slots past a context and table entries past its blocks hold garbage:
    neither may reach the output (blocks of 8: a 16-token tile whose second
    block lies past the context must not read that block's table entry)."""
    lens, Hq, Hkv, D = (5, 17, 40), 8, 2, 128
    pool = sum(workloads.cdiv(n, bs) for n in lens) + 8
    batch = workloads.make_batch("nan", lens, Hq, Hkv, D, bs, pool, True, seed_values=7)
    k, v = batch.k_cache, batch.v_cache
    for b, n in enumerate(lens):
        last = batch.block_tables[b, workloads.cdiv(n, bs) - 1]
        k[last, n % bs or bs:] = 0x7FC0   # NaN
        v[last, n % bs or bs:] = 0x7FC0
    tables = batch.block_tables.copy()
    extra = np.full((len(lens), 3), 10**6, np.int32)
    batch.block_tables = np.concatenate([tables, extra], axis=1)
    batch.new_pos = np.full(len(lens), -1, np.int32)   # no scatter: keep the NaN tails
    db = DeviceBatch(batch)
    for ws in (None, make_workspace(batch)):
        out = torch.empty((3, Hq, D), dtype=torch.float32, device="cuda")
        pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                     max(lens), batch.scale, workspace=ws)
        want = oracle.paged_attention(batch.query, k, v, tables, batch.context_lens, batch.scale)
        assert max_err(out, want) <= ATOL
    assert_clean_status()


def test_decode_empty_and_single_token():
    lens, Hq, Hkv, D, bs = (0, 1, 0, 33), 8, 2, 128, 16
    batch = workloads.make_batch("edge", lens, Hq, Hkv, D, bs, 16, True, seed_values=9)
    db = DeviceBatch(batch)
    for ws in (None, make_workspace(batch)):
        out = torch.full((4, Hq, D), 7.0, dtype=torch.float32, device="cuda")
        pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                     max(lens), batch.scale, workspace=ws)
        o = out.cpu().numpy()
        assert np.all(o[0] == 0) and np.all(o[2] == 0)
        # one token: the output is that token's V row, exactly
        v0 = workloads.bf16_to_f32(batch.v_cache[batch.block_tables[1, 0], 0])  # [Hkv, D]
        for h in range(Hq):
            assert np.array_equal(o[1, h], v0[h // 4])
        want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                      batch.context_lens, batch.scale)
        assert max_err(out, want) <= ATOL
    assert_clean_status()


def test_decode_bf16_output():
    batch = workloads.make_batch("bf16out", (100, 513), 32, 8, 128, 16, 64, True, seed_values=4)
    db = DeviceBatch(batch)
    out = run_step(db, workspace=make_workspace(batch), out_dtype=torch.bfloat16)
    want, _, _ = oracle_step(batch)
    g = out.float().cpu().numpy()
    # rounding the output to bf16 adds at most half an ulp: 2^-8 relative
    assert np.all(np.abs(g - want) <= ATOL + np.abs(want) * 2.0 ** -8)
    assert_clean_status()


# ---------------------------------------------------------------------------
# split-K partitions and the log-sum-exp merge
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bs,ps", [(16, 512), (8, 64), (32, 96), (16, 48), (8, 24), (4, 32), (1, 48)])
def test_splitk_partitions_and_merge(bs, ps):
    lens = (1, 100, 511, 512, 513, 1500)
    Hq, Hkv, D = 16, 4, 128
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("splitk", lens, Hq, Hkv, D, bs, need + 5, True, seed_values=ps + bs)
    db = DeviceBatch(batch)
    P = workloads.cdiv(max(lens), ps)
    tmp = torch.full((len(lens), Hq, P, D), 3.0, dtype=torch.float32, device="cuda")
    ml = torch.full((len(lens), Hq, P), 3.0, dtype=torch.float32, device="cuda")
    es = torch.full((len(lens), Hq, P), 3.0, dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk(tmp, ml, es, ps, db.query, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, max(lens), batch.scale)
    po, pm, psum = oracle.paged_attention_partitions(batch.query, batch.k_cache, batch.v_cache,
                                                     batch.block_tables, batch.context_lens,
                                                     batch.scale, ps, P)
    assert max_err(tmp, po) <= ATOL
    ml_h, es_h = ml.cpu().numpy().astype(np.float64), es.cpu().numpy().astype(np.float64)
    empty = psum == 0
    assert np.array_equal(np.isneginf(ml_h), empty) and np.all(es_h[empty] == 0)
    live = ~empty
    # the partition's log-sum-exp, max + log(sum), is what the merge consumes
    lse_got = ml_h[live] + np.log(es_h[live])
    lse_want = pm[live] + np.log(psum[live])
    assert np.max(np.abs(lse_got - lse_want)) <= 1e-4
    out = torch.empty((len(lens), Hq, D), dtype=torch.float32, device="cuda")
    pa.pa_lse_merge(out, tmp, ml, es, db.context_lens, ps)
    full = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    assert max_err(out, full) <= ATOL
    # the oracle's own merge of the oracle's partitions is the same answer
    assert np.max(np.abs(oracle.lse_merge(po, pm, psum) - full)) < 1e-12
    assert_clean_status()


@pytest.mark.parametrize("num_seqs,hq", [(2, 8), (48, 32)])
def test_lse_merge_few_and_many_rows(num_seqs, hq):
    """pa_lse_merge takes one of two forms by (sequence, head) rows per SM: a
    barrier-free online merge for few rows, shared-memory weights for many.
    Both must give whole-context attention: ragged lengths leave trailing
    partitions empty, and 19 partitions span several batches of eight."""
    rng = np.random.default_rng(num_seqs)
    lens = rng.integers(1, 19 * 64 + 1, size=num_seqs).astype(np.int32)
    lens[0] = 19 * 64
    hkv, d, bs, ps = hq // 4, 128, 16, 64
    need = sum(workloads.cdiv(int(n), bs) for n in lens)
    batch = workloads.make_batch("merge", lens, hq, hkv, d, bs, need + 3, True, seed_values=70 + num_seqs)
    db = DeviceBatch(batch)
    P = workloads.cdiv(int(lens.max()), ps)
    tmp = torch.full((num_seqs, hq, P, d), float("nan"), dtype=torch.float32, device="cuda")
    ml = torch.full((num_seqs, hq, P), float("nan"), dtype=torch.float32, device="cuda")
    es = torch.full((num_seqs, hq, P), float("nan"), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk(tmp, ml, es, ps, db.query, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, int(lens.max()), batch.scale)
    out = torch.empty((num_seqs, hq, d), dtype=torch.float32, device="cuda")
    pa.pa_lse_merge(out, tmp, ml, es, db.context_lens, ps)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    assert max_err(out, want) <= ATOL
    assert_clean_status()


# ---------------------------------------------------------------------------
# scatter and copy: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bf16", [False, True])
def test_reshape_and_cache_bit_exact(bf16):
    rng = np.random.default_rng(21)
    nb, bs, hkv, d, T = 40, 16, 8, 128, 97
    dt = np.uint16 if bf16 else np.float32
    draw = lambda shape: (workloads.bf16_round(rng.standard_normal(shape, dtype=np.float32)) if bf16
                          else rng.standard_normal(shape, dtype=np.float32))
    k, v = draw((nb, bs, hkv, d)), draw((nb, bs, hkv, d))
    key, val = draw((T, hkv, d)), draw((T, hkv, d))
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::10] = -1                 # padding tokens are skipped
    slots[5] = nb * bs + 3           # past the pool: skipped, never written
    kd, vd = to_dev(k), to_dev(v)
    pa.pa_reshape_and_cache(to_dev(key), to_dev(val), kd, vd, torch.from_numpy(slots).cuda())
    ok = slots < nb * bs
    oracle.reshape_and_cache(k, v, key[ok], val[ok], slots[ok])
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert_clean_status()


@pytest.mark.parametrize("bs,dtype", [(16, np.uint16), (32, np.uint16), (8, np.float32)])
def test_copy_blocks_bit_exact(bs, dtype):
    rng = np.random.default_rng(bs)
    nb, hkv, d = 200, 8, 128
    k = rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(np.uint16)
    v = rng.integers(0, 2**16, size=(nb, bs, hkv, d)).astype(np.uint16)
    if dtype == np.float32:
        k = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
        v = rng.standard_normal((nb, bs, hkv, d)).astype(np.float32)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:63], perm[63:126]], axis=1).astype(np.int64)
    kd, vd = to_dev(k), to_dev(v)
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(k, v, pairs)
    assert np.array_equal(to_host_bits(kd), k) and np.array_equal(to_host_bits(vd), v)
    assert_clean_status()


# ---------------------------------------------------------------------------
# the five workloads at full size (decode through the same call bench.py times)
# ---------------------------------------------------------------------------
def test_toy_workload():
    batch = workloads.toy()
    db = DeviceBatch(batch)
    out = run_step(db, workspace=make_workspace(batch))
    want, k_want, v_want = oracle_step(batch)
    assert np.array_equal(to_host_bits(db.k_cache), k_want)
    assert max_err(out, want) <= ATOL
    assert_clean_status()


def test_gqa_workload():
    batch = workloads.gqa()
    db = DeviceBatch(batch)
    out = run_step(db, workspace=make_workspace(batch))
    want, _, _ = oracle_step(batch)
    assert max_err(out, want) <= ATOL
    assert_clean_status()


def test_qwen3_workload():
    batch = workloads.qwen3()
    db = DeviceBatch(batch)
    ws = make_workspace(batch)
    out = run_step(db, workspace=ws)
    want, k_want, v_want = oracle_step(batch)
    # the 16 scattered tokens landed exactly; the rest of the pool is untouched
    assert np.array_equal(to_host_bits(db.k_cache), k_want)
    assert np.array_equal(to_host_bits(db.v_cache), v_want)
    assert max_err(out, want) <= ATOL
    assert_clean_status()


@pytest.mark.parametrize("bs", [4, 8, 16, 32])
def test_long_context_workload(bs):
    batch = workloads.long_context(block_size=bs)
    db = DeviceBatch(batch)
    out = run_step(db, workspace=make_workspace(batch))
    want, _, _ = oracle_step(batch)
    assert max_err(out, want) <= ATOL
    # the explicit 512-token split-K path + merge gives the same answer
    P = workloads.cdiv(batch.max_context_len, 512)
    B, Hq, D = batch.num_seqs, batch.num_heads, batch.head_dim
    tmp = torch.empty((B, Hq, P, D), dtype=torch.float32, device="cuda")
    ml = torch.empty((B, Hq, P), dtype=torch.float32, device="cuda")
    es = torch.empty((B, Hq, P), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk(tmp, ml, es, 512, db.query, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, batch.max_context_len, batch.scale)
    out2 = torch.empty_like(out)
    pa.pa_lse_merge(out2, tmp, ml, es, db.context_lens, 512)
    assert max_err(out2, want) <= ATOL
    assert_clean_status()


@pytest.mark.parametrize("prefix_len,expect_pairs", [(2048, 0), (2064, 63)])
def test_shared_prefix_cow_workload(prefix_len, expect_pairs):
    """64 sequences share a prefix through the block manager (refcount 64);
    each writes its suffix and one decode token, cloning the shared partial
    block first when there is one (copy_blocks), then one decode step."""
    case = workloads.shared_prefix(prefix_len=prefix_len)
    S, bs, hkv, d = len(case.suffix_lens), case.block_size, case.num_kv_heads, case.head_dim
    bm = pa.BlockManager(case.num_blocks, bs)
    model = oracle.BlockManagerModel(case.num_blocks, bs)
    kd = torch.zeros((case.num_blocks, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    k_h = np.zeros((case.num_blocks, bs, hkv, d), np.uint16)
    v_h = np.zeros_like(k_h)
    # prefill of the shared prefix: sequence 0, then forks
    bm.allocate(0, prefix_len)
    model.allocate(0, prefix_len)
    pre_slots = pa.pa_compute_slot_mapping(np.array([bm.block_table(0)], np.int32),
                                           np.zeros(prefix_len, np.int32),
                                           np.arange(prefix_len, dtype=np.int32), bs)
    pa.pa_reshape_and_cache(to_dev(case.prefix_key), to_dev(case.prefix_value), kd, vd,
                            torch.from_numpy(pre_slots).cuda())
    oracle.reshape_and_cache(k_h, v_h, case.prefix_key, case.prefix_value,
                             oracle.slot_mapping([model.block_table(0)], np.zeros(prefix_len, int),
                                                 np.arange(prefix_len), bs))
    for s in range(1, S):
        bm.fork(0, s)
        model.fork(0, s)
    assert bm.stats()["shared_blocks"] == workloads.cdiv(prefix_len, bs)
    # suffix + decode token for every sequence, in sequence order
    pairs, slots, keys, vals = [], [], [], []
    for s in range(S):
        for t in range(case.suffix_key[s].shape[0]):
            slot, src, dst = bm.append_slot(s)
            assert (slot, src, dst) == model.append_slot(s)
            if src >= 0:
                pairs.append((src, dst))
            slots.append(slot)
        keys.append(case.suffix_key[s])
        vals.append(case.suffix_value[s])
    assert len(pairs) == expect_pairs
    if pairs:
        pm = np.array(pairs, np.int64)
        pa.pa_copy_blocks(kd, vd, torch.from_numpy(pm).cuda())
        oracle.copy_blocks(k_h, v_h, pm)
    keys, vals = np.concatenate(keys), np.concatenate(vals)
    slots = np.array(slots, np.int64)
    pa.pa_reshape_and_cache(to_dev(keys), to_dev(vals), kd, vd, torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache(k_h, v_h, keys, vals, slots)
    assert np.array_equal(to_host_bits(kd), k_h) and np.array_equal(to_host_bits(vd), v_h)
    # decode over prefix + suffix + 1 tokens
    lens = np.array([bm.num_tokens(s) for s in range(S)], np.int32)
    assert np.array_equal(lens, prefix_len + case.suffix_lens + 1)
    maxb = max(len(bm.block_table(s)) for s in range(S))
    tables = np.zeros((S, maxb), np.int32)
    for s in range(S):
        t = bm.block_table(s)
        tables[s, :len(t)] = t
    batch = workloads.DecodeBatch("cow", case.query, k_h, v_h, tables, lens, None, None, None, bs,
                                  case.num_heads, hkv, d, case.scale, True)
    ws = make_workspace(batch)
    out = torch.empty((S, case.num_heads, d), dtype=torch.float32, device="cuda")
    pa.pa_decode(out, to_dev(case.query), kd, vd, to_dev(tables), to_dev(lens), int(lens.max()),
                 case.scale, workspace=ws)
    want = oracle.paged_attention(case.query, k_h, v_h, tables, lens, case.scale)
    assert max_err(out, want) <= ATOL
    assert_clean_status()
