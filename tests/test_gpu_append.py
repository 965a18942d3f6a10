"""pa_decode_append: one decode step ("PagedAttention, explained.", procedure
steps 4 and 5) -- each sequence's new token written to position
context_len - 1, then attention over the whole context. The per-partition
tensor-core kernel writes the token itself (the CTA that reads its tile
stores it first); other plans scatter ahead. The result must be the
oracle's (scatter, then attention over the updated cache), the caches bit
for bit, and bit for bit the result of pa_reshape_and_cache + pa_decode, on
every path: cluster and workspace splits, each load mode, the CUDA-core
kernel, the ragged-balanced path, fp16; a refused call writes nothing."""
import numpy as np
import pytest
import torch

import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import (ATOL, DeviceBatch, make_workspace, max_err, new_token_slots, oracle_step,
                       to_host_bits)

pytestmark = pytest.mark.gpu

CASES = [
    # lens, Hq, Hkv, D, block size, f16, workspace
    ((1, 2, 15, 16, 17, 100, 333), 8, 2, 128, 16, False, False),   # cluster merge
    ((3000, 4000), 16, 4, 128, 16, False, True),                   # wide split + merge kernel
    ((1, 7, 8, 9, 64, 250), 16, 4, 128, 8, False, True),           # two blocks per tile
    ((19, 90, 300), 8, 2, 128, 4, True, True),                     # bulk row copies, fp16
    ((40, 90), 8, 2, 64, 12, False, True),                         # CUDA-core kernel: scatter launched first
    ((0, 5, 33, 0, 200, 16), 16, 4, 128, 32, False, False),         # empty sequences write nothing
    ((1, 255, 256, 257, 600), 8, 2, 128, 256, False, True),          # new tokens on both sides of a 256-token block boundary
]


def run_append(db, ws, out_dtype=torch.float32):
    b = db.h
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=out_dtype, device="cuda")
    pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, b.max_context_len, b.scale, workspace=ws)
    return out


def run_separate(db, ws, out_dtype=torch.float32):
    b = db.h
    slots = torch.from_numpy(new_token_slots(b)).cuda()
    pa.pa_reshape_and_cache(db.new_key, db.new_value, db.k_cache, db.v_cache, slots)
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=out_dtype, device="cuda")
    pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens, b.max_context_len,
                 b.scale, workspace=ws)
    return out


def bits(t):
    return t.cpu().view(torch.int16).numpy() if t.element_size() == 2 else to_host_bits(t)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_matches_oracle_and_separate_calls(case):
    lens, hq, hkv, d, bs, f16, use_ws = CASES[case]
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("append", lens, hq, hkv, d, bs, need + 9, not f16, seed_values=900 + case,
                                 f16=f16)
    batch.new_pos = np.array([n - 1 if n > 0 else -1 for n in lens], np.int32)   # the new token: position len - 1
    db = DeviceBatch(batch)
    ws = make_workspace(batch) if use_ws else None
    out = run_append(db, ws)
    want, k_want, v_want = oracle_step(batch)
    assert np.array_equal(bits(db.k_cache), np.ascontiguousarray(k_want).view(np.int16))
    assert np.array_equal(bits(db.v_cache), np.ascontiguousarray(v_want).view(np.int16))
    assert max_err(out, want) <= ATOL
    # the same two calls made separately, on a fresh copy of the inputs
    db2 = DeviceBatch(batch)
    out2 = run_separate(db2, make_workspace(batch) if use_ws else None)
    assert torch.equal(out, out2)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0


def test_append_balanced_and_in_a_graph():
    rng = np.random.default_rng(950)
    lens = rng.integers(1, 600, size=160).astype(np.int32)
    need = sum(workloads.cdiv(int(n), 16) for n in lens)
    batch = workloads.make_batch("append_bal", lens, 32, 8, 128, 16, need + 9, True, seed_values=951)
    assert pa.pa_decode_plan(160, 32, 8, 128, 16, int(lens.max()), with_workspace=True)["balanced"]
    db = DeviceBatch(batch)
    ws = make_workspace(batch)
    out = torch.empty((160, 32, 128), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache,
                            db.block_tables, db.context_lens, batch.max_context_len, batch.scale, workspace=ws)
    torch.cuda.synchronize()
    want, _, _ = oracle_step(batch)
    assert max_err(out, want) <= ATOL
    # captured and replayed: the scatter rewrites the same values, the decode gives the same output
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache,
                            db.block_tables, db.context_lens, batch.max_context_len, batch.scale, workspace=ws)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert max_err(out, want) <= ATOL
    assert pa.pa_device_status(clear=True) == 0


def test_append_refuses_before_launching():
    """A shape the decode refuses (8 query heads over 3 KV heads) launches
    nothing: the scatter must not have written its rows either."""
    batch = workloads.make_batch("append_bad", (10, 20), 8, 2, 128, 16, 8, True, seed_values=960)
    db = DeviceBatch(batch)
    before = bits(db.k_cache).copy()
    out = torch.empty((2, 8, 128), dtype=torch.float32, device="cuda")
    lib = pa.load_library()
    args = [out.data_ptr(), pa.PA_F32, db.query.data_ptr(), pa.PA_BF16, db.new_key.data_ptr(),
            db.new_value.data_ptr(), db.k_cache.data_ptr(), db.v_cache.data_ptr(), pa.PA_BF16,
            db.block_tables.data_ptr(), db.context_lens.data_ptr(), 2, 8, 3, 128, 16,
            int(db.block_tables.shape[1]), 8, 20, 0.1, None, 0, torch.cuda.current_stream().cuda_stream]
    assert lib.pa_decode_append(*args) == pa.PA_ERR_INVALID_ARG
    # a split that needs a workspace, called with a null one: refused, nothing written either
    long_batch = workloads.make_batch("append_ws", (3000, 4000), 16, 4, 128, 16, 450, True, seed_values=961)
    ldb = DeviceBatch(long_batch)
    lbefore = bits(ldb.k_cache).copy()
    lout = torch.empty((2, 16, 128), dtype=torch.float32, device="cuda")
    assert not pa.pa_decode_plan(2, 16, 4, 128, 16, 4000, with_workspace=True)["cluster_merge"]
    status = lib.pa_decode_append(lout.data_ptr(), pa.PA_F32, ldb.query.data_ptr(), pa.PA_BF16,
                                  ldb.new_key.data_ptr(), ldb.new_value.data_ptr(), ldb.k_cache.data_ptr(),
                                  ldb.v_cache.data_ptr(), pa.PA_BF16, ldb.block_tables.data_ptr(),
                                  ldb.context_lens.data_ptr(), 2, 16, 4, 128, 16, int(ldb.block_tables.shape[1]),
                                  450, 4000, 0.1, None, 1, torch.cuda.current_stream().cuda_stream)
    assert status == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert np.array_equal(bits(db.k_cache), before)
    assert np.array_equal(bits(ldb.k_cache), lbefore)


# ---------------------------------------------------------------------------
# The step bench.py times, at full size: the bench's own batches (two
# disjoint batches of sequences in one pool), its workspace and plan, the
# steps alternating between the two batches inside one CUDA graph. Caches bit
# for bit and both batches' outputs against the oracle.
# ---------------------------------------------------------------------------
FULL = [
    # bench config, plan the step must take (checked, so the test keeps
    # covering the launch configuration the bench reports)
    ("qwen3", dict(tensor_cores=1, cluster_merge=1, balanced=0, kernel_launches=1)),   # 8-CTA cluster merge
    ("long", dict(tensor_cores=1, cluster_merge=0, balanced=0, kernel_launches=2)),    # workspace split + merge
    ("gqa", dict(tensor_cores=1, balanced=1, kernel_launches=2)),                       # ragged-balanced
]


@pytest.mark.parametrize("config,plan_keys", FULL, ids=[c for c, _ in FULL])
def test_append_full_size_bench_step(config, plan_keys):
    import bench
    import oracle
    from gpu_cases import to_dev

    batch, _ = bench.build_workload(config, 0, 2)
    nb = bench.per_batch(config)
    hq, hkv, d, bs = batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size
    k_cache, v_cache = to_dev(batch.k_cache), to_dev(batch.v_cache)
    views = []
    for c in range(2):
        sl = slice(c * nb, (c + 1) * nb)
        lens = batch.context_lens[sl]
        views.append(dict(sl=sl, query=to_dev(batch.query[sl]), tables=to_dev(batch.block_tables[sl]),
                          lens=to_dev(lens), key=to_dev(batch.new_key[sl]), value=to_dev(batch.new_value[sl]),
                          max_len=int(lens.max()),
                          out=torch.full((nb, hq, d), float("nan"), dtype=torch.float32, device="cuda")))
    for v in views:
        plan = pa.pa_decode_plan(nb, hq, hkv, d, bs, v["max_len"], with_workspace=True)
        assert {k: plan[k] for k in plan_keys} == plan_keys, plan
    ws_bytes = max(pa.pa_decode_workspace_size(nb, hq, hkv, d, bs, v["max_len"]) for v in views)
    # the bench leaves its workspace as the previous step left it; start from garbage here
    ws = torch.randint(0, 256, (max(ws_bytes, 1),), dtype=torch.uint8, device="cuda")

    def step(i):
        v = views[i % 2]
        pa.pa_decode_append(v["out"], v["query"], v["key"], v["value"], k_cache, v_cache, v["tables"],
                            v["lens"], v["max_len"], batch.scale, workspace=ws)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step(0)
        step(1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for i in range(4):
            step(i)
    for v in views:
        v["out"].fill_(float("nan"))
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0

    # oracle: every sequence's new token at position len - 1, then fp64 attention per batch
    k_want, v_want = batch.k_cache.copy(), batch.v_cache.copy()
    seq = np.arange(batch.num_seqs)
    slots = oracle.slot_mapping(batch.block_tables, seq, batch.context_lens - 1, bs)
    oracle.reshape_and_cache(k_want, v_want, batch.new_key, batch.new_value, slots)
    assert np.array_equal(to_host_bits(k_cache), k_want)
    assert np.array_equal(to_host_bits(v_cache), v_want)
    for v in views:
        sl = v["sl"]
        want = oracle.paged_attention(batch.query[sl], k_want, v_want, batch.block_tables[sl],
                                      batch.context_lens[sl], batch.scale)
        err = max_err(v["out"], want)
        assert err <= ATOL, (config, err)
