"""Failure detection on the GPU, without a fault: a bounded wait runs out.

Every wait of the decode kernels on an asynchronous copy is bounded; past its
limit the kernel records PA_ERR_TIMEOUT in the device status word, stops and
returns. pa_check_wait_timeout runs that path in a CTA laid out as the
kernels' pipeline whose stage is armed for a copy that is never issued, with
the limit cut to a millisecond. The host must read PA_ERR_TIMEOUT once, the
word must clear, and the device must stay usable: a decode right after gives
the oracle's answer and leaves the word at 0."""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, max_err

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0
    t0 = time.perf_counter()
    pa.pa_check_wait_timeout(1000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, elapsed          # the 1 ms limit, not the kernels' 2 s, ended the waits
    assert pa.pa_device_status(clear=True) == pa.PA_ERR_TIMEOUT
    assert pa.pa_device_status(clear=True) == 0    # cleared
    # the context is still usable
    batch = workloads.make_batch("after_timeout", (33, 700), 16, 4, 128, 16, 64, True, seed_values=77)
    db = DeviceBatch(batch)
    out = torch.empty((2, 16, 128), dtype=torch.float32, device="cuda")
    pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                 batch.max_context_len, batch.scale)
    torch.cuda.synchronize()
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    assert max_err(out, want) <= ATOL
    assert pa.pa_device_status(clear=True) == 0

