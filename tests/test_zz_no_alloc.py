"""pa_decode_static_scratch: decode for callers that cannot allocate device memory.

Such callers (an engine whose device memory is all reserved up front by its
own allocator, or a plugin interface that hands over only inputs and outputs)
cannot pass pa_decode a workspace. This entry point merges a context split
inside a thread-block cluster when the split fits one, and through a fixed
scratch array built into the library when it is wider. These tests run it
through the C ABI and compare it with the fp64 oracle, and with pa_decode
given a workspace, on two calls in a row (the scratch keeps the previous
call's contents), and check that a problem too large for the fixed scratch is
refused before any launch. This file is collected last so that a failure here
stops a -x run only after every other test has run; it also passes alone in
a fresh process (its first call does the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
from paged_kv_cache_121_gb300 import _lib
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, max_err

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20   # PA_STATIC_SCRATCH_BYTES in include/pa.h

CASES = [
    # lens, Hq, Hkv, D, block_size, merge: long contexts so that the decode splits
    ((700, 3000, 1500, 4164), 32, 8, 128, 16, "scratch"),
    ((9000, 17), 64, 8, 128, 32, "scratch"),
    ((2000, 1999, 1500, 37, 2000, 1, 640, 1024, 2000, 1777, 3, 999, 1200, 2000, 15, 16), 32, 8, 128, 16,
     "cluster"),
]


def call_static(lib, out, db, batch, stream):
    B, Hq, D = out.shape
    return lib.pa_decode_static_scratch(
        ctypes.c_void_p(out.data_ptr()), pa.PA_F32, ctypes.c_void_p(db.query.data_ptr()),
        pa.PA_BF16, ctypes.c_void_p(db.k_cache.data_ptr()), ctypes.c_void_p(db.v_cache.data_ptr()),
        pa.PA_BF16, ctypes.c_void_p(db.block_tables.data_ptr()),
        ctypes.c_void_p(db.context_lens.data_ptr()), B, Hq, batch.num_kv_heads, D, batch.block_size,
        batch.max_blocks_per_seq, batch.num_blocks, batch.max_context_len, batch.scale, stream)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_oracle_and_workspace_decode(case):
    lens, Hq, Hkv, D, bs, merge = CASES[case]
    plan = pa.pa_decode_plan(len(lens), Hq, Hkv, D, bs, max(lens), with_workspace=True)
    assert not plan["balanced"] and plan["num_splits"] > 1, plan
    if merge == "cluster":
        assert plan["cluster_merge"] == 1, plan
    else:
        assert plan["cluster_merge"] == 0 and 0 < plan["workspace_bytes"] <= STATIC_SCRATCH_BYTES, plan
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("noalloc", lens, Hq, Hkv, D, bs, need + 11, True,
                                 seed_values=900 + case, seed_blocks=910 + case)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    db = DeviceBatch(batch)
    ref = torch.empty((len(lens), Hq, D), dtype=torch.float32, device="cuda")
    pa.pa_decode(ref, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                 batch.max_context_len, batch.scale, workspace=make_workspace(batch))
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        st = call_static(lib, out, db, batch, stream)
        assert st == pa.PA_OK, (call, st)
        torch.cuda.synchronize()
        err = max_err(out, want)
        assert err <= ATOL, (call, err)
        assert float((out - ref).abs().max()) <= ATOL, call
    assert pa.pa_device_status(clear=True) == 0


@pytest.mark.parametrize("merge", ["scratch", "cluster"])
def test_static_scratch_fp16(merge):
    """fp16 query, caches and output, through the scratch and through a cluster."""
    lens = (3000, 4164, 17, 900) if merge == "scratch" else (2000, 1999, 37, 1500, 2000, 64, 1024, 1777) * 2
    Hq, Hkv, D, bs = 32, 8, 128, 16
    plan = pa.pa_decode_plan(len(lens), Hq, Hkv, D, bs, max(lens), kv_dtype=pa.PA_F16, with_workspace=True)
    assert plan["cluster_merge"] == (1 if merge == "cluster" else 0) and plan["num_splits"] > 1, plan
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("noalloc16", lens, Hq, Hkv, D, bs, need + 5, False, seed_values=930, f16=True)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    db = DeviceBatch(batch)
    out = torch.full((len(lens), Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    pa.pa_decode_static_scratch(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                batch.max_context_len, batch.scale)
    torch.cuda.synchronize()
    g = out.float().cpu().numpy()
    # rounding the output to fp16 adds at most half an ulp: 2^-11 relative
    assert np.all(np.abs(g - want) <= ATOL + np.abs(want) * 2.0 ** -11)
    assert pa.pa_device_status(clear=True) == 0


def test_static_scratch_refuses_problem_larger_than_scratch():
    """A shape whose split (as pa_decode_plan reports it on this GPU) needs
    more than the fixed scratch is refused before any pointer is touched:
    every pointer here is null."""
    lib = _lib.load()
    # few sequences, many query heads per KV head, long contexts: a wide
    # split (beyond a cluster) whose partials grow with the GPU's SM count
    candidates = [(4, 64, 4, 128, 16, 32768), (2, 128, 2, 128, 16, 65536), (1, 256, 4, 128, 16, 131072)]
    for B, Hq, Hkv, D, bs, ctx in candidates:
        plan = pa.pa_decode_plan(B, Hq, Hkv, D, bs, ctx, with_workspace=True)
        if plan["balanced"] or plan["cluster_merge"] or plan["workspace_bytes"] <= STATIC_SCRATCH_BYTES:
            continue
        st = lib.pa_decode_static_scratch(None, pa.PA_F32, None, pa.PA_BF16, None, None, pa.PA_BF16,
                                          None, None, B, Hq, Hkv, D, bs, ctx // bs, 200000, ctx,
                                          0.088, None)
        assert st == pa.PA_ERR_WORKSPACE, (B, Hq, Hkv, plan)
        return
    pytest.skip("no candidate shape splits wider than the scratch holds on a GPU with this few SMs")
