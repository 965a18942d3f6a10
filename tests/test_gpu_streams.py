"""Calls on several streams at once. The library keeps no per-call state on
the host or the device (plans are recomputed per call; workspaces belong to
the caller), so decodes of different batches issued on different streams,
interleaved and unsynchronised, each give the oracle's answer. Covers the
cluster, workspace-split and ragged-balanced plans and pa_decode_append."""
import numpy as np
import pytest
import torch

import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, max_err, oracle_step

pytestmark = pytest.mark.gpu


def batch_for(kind, seed):
    if kind == "cluster":        # 16 sequences: split inside a cluster
        lens = np.random.default_rng(seed).integers(300, 900, size=16)
    elif kind == "split":        # 2 long sequences: split through the workspace
        lens = (3000, 4000)
    else:                        # 140 ragged sequences: the balanced plan
        lens = np.random.default_rng(seed).integers(1, 400, size=140)
    need = sum(workloads.cdiv(int(n), 16) for n in lens)
    return workloads.make_batch(kind, lens, 32, 8, 128, 16, need + 5, True, seed_values=seed)


def test_interleaved_streams():
    kinds = ["cluster", "split", "balanced"]
    batches = [batch_for(k, 40 + i) for i, k in enumerate(kinds)]
    dbs = [DeviceBatch(b) for b in batches]
    wss = [make_workspace(b) for b in batches]
    outs = [torch.empty((b.num_seqs, 32, 128), dtype=torch.float32, device="cuda") for b in batches]
    streams = [torch.cuda.Stream() for _ in batches]
    plans = [pa.pa_decode_plan(b.num_seqs, 32, 8, 128, 16, b.max_context_len, with_workspace=True) for b in batches]
    assert plans[0]["cluster_merge"] and not plans[1]["cluster_merge"] and plans[2]["balanced"]
    torch.cuda.synchronize()
    # the step (new token written, then the decode) once per batch, then plain decodes, all interleaved
    for rep in range(4):
        for db, b, ws, out, s in zip(dbs, batches, wss, outs, streams):
            with torch.cuda.stream(s):
                if rep == 0:
                    pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache,
                                        db.block_tables, db.context_lens, b.max_context_len, b.scale, workspace=ws)
                else:
                    pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                                 b.max_context_len, b.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0
    for b, out in zip(batches, outs):
        want, _, _ = oracle_step(b)
        assert max_err(out, want) <= ATOL
