"""pa_decode_static_scratch: decode for callers that cannot allocate device memory.

Such callers (an engine whose device memory is all reserved up front by its
own allocator, or a plugin interface that hands over only inputs and outputs)
cannot pass pa_decode a workspace. This entry point merges a context split
through a fixed scratch array built into the library instead. These tests run
it through the C ABI and compare it with pa_decode given a workspace, on two
calls in a row (the scratch keeps the previous call's contents), and check
that a problem too large for the fixed scratch is refused before any launch.
This file is collected last so that a failure here stops a -x run only after
every other test has run; it also passes alone in a fresh process (its first
call does the per-device set-up).
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_121_gb300 as pa
from paged_kv_cache_121_gb300 import _lib
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace

pytestmark = pytest.mark.gpu

CASES = [
    # lens, Hq, Hkv, D, block_size: long contexts so that the decode splits
    ((700, 3000, 1500, 4164), 32, 8, 128, 16),
    ((9000, 17), 64, 8, 128, 32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_workspace_decode(case):
    lens, Hq, Hkv, D, bs = CASES[case]
    need = sum(workloads.cdiv(n, bs) for n in lens)
    batch = workloads.make_batch("noalloc", lens, Hq, Hkv, D, bs, need + 11, True,
                                 seed_values=900 + case, seed_blocks=910 + case)
    db = DeviceBatch(batch)
    ref = torch.empty((len(lens), Hq, D), dtype=torch.float32, device="cuda")
    pa.pa_decode(ref, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                 batch.max_context_len, batch.scale, workspace=make_workspace(batch))
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        st = lib.pa_decode_static_scratch(
            ctypes.c_void_p(out.data_ptr()), pa.PA_F32, ctypes.c_void_p(db.query.data_ptr()),
            pa.PA_BF16, ctypes.c_void_p(db.k_cache.data_ptr()), ctypes.c_void_p(db.v_cache.data_ptr()),
            pa.PA_BF16, ctypes.c_void_p(db.block_tables.data_ptr()),
            ctypes.c_void_p(db.context_lens.data_ptr()), len(lens), Hq, Hkv, D, bs,
            batch.max_blocks_per_seq, batch.num_blocks, batch.max_context_len, batch.scale, stream)
        assert st == pa.PA_OK, (call, st)
        torch.cuda.synchronize()
        err = float((out - ref).abs().max())
        assert err <= ATOL, (call, err)
    assert pa.pa_device_status(clear=True) == 0


STATIC_SCRATCH_BYTES = 8 << 20   # PA_STATIC_SCRATCH_BYTES in include/pa.h


def test_static_scratch_refuses_problem_larger_than_scratch():
    lib = _lib.load()
    # 4 sequences of 32k tokens with 64 query heads over 4 KV heads: the
    # decode splits each context many ways and its partials need more than
    # the fixed scratch, so the call is refused before any pointer is touched
    shape = dict(B=4, Hq=64, Hkv=4, D=128, bs=16, ctx=32768)
    need = pa.pa_decode_workspace_size(shape["B"], shape["Hq"], shape["Hkv"], shape["D"],
                                       shape["bs"], shape["ctx"])
    assert need > STATIC_SCRATCH_BYTES
    st = lib.pa_decode_static_scratch(None, pa.PA_F32, None, pa.PA_BF16, None, None, pa.PA_BF16,
                                      None, None, shape["B"], shape["Hq"], shape["Hkv"], shape["D"],
                                      shape["bs"], shape["ctx"] // shape["bs"], 200000, shape["ctx"],
                                      0.088, None)
    assert st == pa.PA_ERR_WORKSPACE
