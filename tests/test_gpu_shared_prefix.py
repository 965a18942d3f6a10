"""Shared-prefix decode (pa_decode_shared_prefix) against the fp64 oracle:
the shared blocks read once for the batch, the rest per sequence, merged by
log-sum-exp, must give plain paged attention ("PagedAttention: KV cache
virtual memory", "Copy-on-write: when two requests share a prefix"; "Paged
Attention: Virtual Memory for the KV Cache", "Sharing a prefix: one copy for
many requests")."""
import json
import os
import subprocess
import sys

if __name__ == "__main__":   # the child process: the repo root, as conftest gives pytest
    sys.path[:0] = [os.path.dirname(os.path.dirname(os.path.abspath(__file__)))]

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, max_err, to_dev

pytestmark = pytest.mark.gpu


def run_shared(db, shared_blocks, out_dtype=torch.float32, workspace=None):
    b = db.h
    n = pa.pa_decode_shared_prefix_workspace_size(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim,
                                                  b.block_size, b.max_context_len, shared_blocks)
    ws = workspace if workspace is not None else torch.full((max(n, 1),), 0xFF, dtype=torch.uint8,
                                                             device="cuda")
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=out_dtype, device="cuda")
    pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                               b.max_context_len, shared_blocks, b.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0
    return out


def oracle_out(b):
    return oracle.paged_attention(b.query, b.k_cache, b.v_cache, b.block_tables, b.context_lens, b.scale)


CASES = [
    # shared_blocks, suffix lengths, Hq, Hkv, D, block_size
    (10, (0, 7, 40, 16, 33), 32, 8, 128, 16),
    (3, (1, 100, 64, 2), 16, 4, 64, 32),
    (7, (0, 20, 9), 8, 2, 128, 8),                  # blocks of 8, odd count: 48 shared tokens in tiles
    (5, (3, 50, 17, 90), 64, 2, 128, 16),           # G = 32: two head tiles
    (4, (5, 0, 77), 8, 8, 64, 16),                  # G = 1
    (2, tuple(range(0, 40)), 8, 2, 128, 32),        # 40 sequences x 4 heads: 160 rows, three row groups
    (6, (0, 0, 0), 16, 4, 128, 16),                 # nothing past the prefix
    (1, (300,), 32, 8, 128, 128),                   # one sequence, one large block shared
    (9, (12, 250, 31), 24, 12, 128, 64),            # 12 KV heads
    (4, (1000, 2000, 5, 700), 32, 8, 128, 16),      # long rests: split, partitions merged by the merge kernel
    (2, (10, 300, 0), 16, 4, 128, 256),             # the largest blocks: 512 shared tokens in two blocks
    (3, tuple(range(5, 75)), 12, 2, 128, 16),       # G = 6: four row groups of 21 sequences (126 rows)
    (2, tuple(range(0, 70)), 32, 8, 64, 32),        # D 64, three row groups, two per CTA: the second pair holds one
    (2, (5, 40, 0), 128, 1, 128, 16),               # G = 128: one sequence per row group, a half pair
    (3, (7, 100), 64, 1, 64, 32),                   # G = 64: two sequences per row group
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_shared_prefix_matches_oracle(case):
    nsh, suffix, hq, hkv, d, bs = CASES[case]
    batch = workloads.shared_prefix_batch("sp", nsh, suffix, hq, hkv, d, bs, seed_values=800 + case,
                                          seed_blocks=900 + case)
    db = DeviceBatch(batch)
    want = oracle_out(batch)
    out = run_shared(db, nsh)
    assert max_err(out, want) <= ATOL
    # the same as the plain paged decode of the same batch (both within the bound of the oracle)
    ref = torch.empty_like(out)
    n = pa.pa_decode_workspace_size(batch.num_seqs, hq, hkv, d, bs, batch.max_context_len)
    pa.pa_decode(ref, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                 batch.max_context_len, batch.scale,
                 workspace=torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda"))
    assert float((out - ref).abs().max()) <= 2 * ATOL


def test_shared_prefix_fewer_blocks_than_shared_and_bf16_out():
    """Declaring fewer shared blocks than the rows share is still exact; so is
    zero (the plain decode); bf16 output rounds once."""
    batch = workloads.shared_prefix_batch("sp", 12, (5, 60, 3), 32, 8, 128, 16, seed_values=820)
    db = DeviceBatch(batch)
    want = oracle_out(batch)
    for nsh in (12, 5, 1, 0):
        assert max_err(run_shared(db, nsh), want) <= ATOL
    g = run_shared(db, 12, out_dtype=torch.bfloat16).float().cpu().numpy()
    assert np.all(np.abs(g - want) <= ATOL + np.abs(want) * 2.0 ** -8)


def test_shared_prefix_workspace_is_reusable_and_required():
    batch = workloads.shared_prefix_batch("sp", 16, (10, 90, 33, 0), 32, 8, 128, 16, seed_values=821)
    db = DeviceBatch(batch)
    n = pa.pa_decode_shared_prefix_workspace_size(4, 32, 8, 128, 16, batch.max_context_len, 16)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    a = run_shared(db, 16, workspace=ws)
    b = run_shared(db, 16, workspace=ws)
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    with pytest.raises(pa.PAError):
        pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                   batch.max_context_len, 16, batch.scale, ws[: n // 2])
    with pytest.raises(pa.PAError):     # more shared blocks than a table row holds
        pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                   batch.max_context_len, batch.max_blocks_per_seq + 1, batch.scale, ws)


@pytest.mark.parametrize("prefix_len", [2048, 2064])
def test_shared_prefix_cow_workload(prefix_len):
    """The copy-on-write workload: 64 sequences forked from one prefix through
    the block manager, suffixes U[0, 256] and one decode token each; the
    shared full blocks (64 of 32 tokens) are read once for the batch."""
    case = workloads.shared_prefix(prefix_len=prefix_len)
    S, bs, hkv, d = len(case.suffix_lens), case.block_size, case.num_kv_heads, case.head_dim
    bm = pa.BlockManager(case.num_blocks, bs)
    k_h = np.zeros((case.num_blocks, bs, hkv, d), np.uint16)
    v_h = np.zeros_like(k_h)
    bm.allocate(0, prefix_len)
    oracle.reshape_and_cache(k_h, v_h, case.prefix_key, case.prefix_value,
                             oracle.slot_mapping([bm.block_table(0)], np.zeros(prefix_len, int),
                                                 np.arange(prefix_len), bs))
    for s in range(1, S):
        bm.fork(0, s)
    pairs, slots, keys, vals = [], [], [], []
    for s in range(S):
        for _ in range(case.suffix_key[s].shape[0]):
            slot, src, dst = bm.append_slot(s)
            if src >= 0:
                pairs.append((src, dst))
            slots.append(slot)
        keys.append(case.suffix_key[s])
        vals.append(case.suffix_value[s])
    if pairs:
        oracle.copy_blocks(k_h, v_h, np.array(pairs, np.int64))
    oracle.reshape_and_cache(k_h, v_h, np.concatenate(keys), np.concatenate(vals), np.array(slots, np.int64))
    lens = np.array([bm.num_tokens(s) for s in range(S)], np.int32)
    maxb = max(len(bm.block_table(s)) for s in range(S))
    tables = np.zeros((S, maxb), np.int32)
    for s in range(S):
        t = bm.block_table(s)
        tables[s, :len(t)] = t
    shared = prefix_len // bs                      # full blocks every row still shares
    assert all(np.array_equal(tables[s, :shared], tables[0, :shared]) for s in range(S))
    batch = workloads.DecodeBatch("cow", case.query, k_h, v_h, tables, lens, None, None, None, bs,
                                  case.num_heads, hkv, d, case.scale, True)
    db = DeviceBatch(batch)
    out = run_shared(db, shared)
    assert max_err(out, oracle_out(batch)) <= ATOL


def test_shared_prefix_negative_scale():
    """A negative softmax scale (the largest scaled score then comes from the
    smallest raw one), both passes, against the oracle."""
    for d, seed in ((128, 870), (64, 871)):
        batch = workloads.shared_prefix_batch("neg", 12, tuple(range(0, 300, 7)), 32, 8, d, 16, seed_values=seed)
        batch.scale = -0.7 / np.sqrt(d)
        out = run_shared(DeviceBatch(batch), 12)
        assert max_err(out, oracle_out(batch)) <= ATOL


def test_shared_prefix_in_a_cuda_graph_matches_eager():
    """The call's three kernels (rest-of-context decode, prefix pass launched
    as its programmatic dependent, merge) captured into a CUDA graph (as a
    serving loop would) and replayed give the eager result."""
    batch = workloads.shared_prefix_batch("sp", 32, tuple(range(5, 400, 25)), 32, 8, 128, 32, seed_values=830)
    db = DeviceBatch(batch)
    n = pa.pa_decode_shared_prefix_workspace_size(batch.num_seqs, 32, 8, 128, 32, batch.max_context_len, 32)
    ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
    eager = run_shared(db, 32, workspace=ws)
    out = torch.zeros_like(eager)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                   batch.max_context_len, 32, batch.scale, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                   batch.max_context_len, 32, batch.scale, ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert max_err(out, oracle_out(batch)) <= ATOL
    assert pa.pa_device_status(clear=True) == 0


def child_cases():
    """Three batches through pa_decode_shared_prefix under the knobs the parent
    set: head_dim 128 with 24 and with 80 sequences (one row group per CTA,
    or two under PA_PREFIX_GROUPS=2), and head_dim 64 with 80 (two)."""
    errs = []
    for seed, suffix, d in ((850, tuple(range(3, 27)), 128), (851, tuple(range(0, 80)), 128),
                            (852, tuple(range(0, 80)), 64)):
        batch = workloads.shared_prefix_batch("knob", 40, suffix, 32, 8, d, 32, seed_values=seed)
        db = DeviceBatch(batch)
        n = pa.pa_decode_shared_prefix_workspace_size(batch.num_seqs, 32, 8, d, 32, batch.max_context_len, 40)
        ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
        out = torch.empty((batch.num_seqs, 32, d), dtype=torch.float32, device="cuda")
        pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                   batch.max_context_len, 40, batch.scale, ws)
        torch.cuda.synchronize()
        errs.append(max_err(out, oracle_out(batch)))
    print(json.dumps({"errs": errs, "status": pa.pa_device_status(clear=True)}))


KNOBS = {
    # the smallest ring budget and few prefix CTAs, so that each CTA streams many
    # tiles through its ring: a ring of one stage would wait on itself (tile
    # i + 1's Q.K^T is issued before tile i's P.V frees its stage), so the
    # tcgen05 pass takes two stages at least whatever the budget
    "smallest_ring": {"PA_DECODE_RING_KB": "16", "PA_PREFIX_CTAS": "16"},
    "smallest_ring_two_groups": {"PA_DECODE_RING_KB": "16", "PA_PREFIX_CTAS": "16", "PA_PREFIX_GROUPS": "2"},
    # the other orders of the two passes: the decode first, the prefix pass as
    # its programmatic dependent; or one after the other
    "rest_first": {"PA_PREFIX_ORDER": "rest"},
    "serial": {"PA_PREFIX_OVERLAP": "0"},
}


@pytest.mark.parametrize("knobs", sorted(KNOBS))
def test_shared_prefix_under_knobs(knobs):
    """Knobs are read once per process: a child process runs the batches."""
    env = dict(os.environ, **KNOBS[knobs])
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == 0 and max(res["errs"]) <= ATOL, res


if __name__ == "__main__" and sys.argv[1:] == ["child"]:
    child_cases()
