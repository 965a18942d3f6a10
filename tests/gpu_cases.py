"""Helpers shared by the GPU tests: move seeded inputs to the device, run the
CUDA path through the C ABI, and run the oracle on the same inputs."""
import math

import numpy as np
import torch

import oracle
import paged_kv_cache_121_gb300 as pa

ATOL = 2e-3   # max abs error vs the fp64 oracle (bf16 K/V, fp32 accumulation)


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


class DeviceBatch:
    """A workloads.DecodeBatch on the device."""

    def __init__(self, batch):
        self.h = batch
        self.query = to_dev(batch.query)
        self.k_cache = to_dev(batch.k_cache)
        self.v_cache = to_dev(batch.v_cache)
        self.block_tables = to_dev(batch.block_tables)
        self.context_lens = to_dev(batch.context_lens)
        self.new_key = to_dev(batch.new_key) if batch.new_key is not None else None
        self.new_value = to_dev(batch.new_value) if batch.new_value is not None else None


def new_token_slots(batch) -> np.ndarray:
    """Slots of each sequence's newest token, from libpa's host slot map."""
    seq = np.arange(batch.num_seqs, dtype=np.int32)
    return pa.pa_compute_slot_mapping(batch.block_tables, seq, batch.new_pos, batch.block_size)


def run_step(db: DeviceBatch, workspace=None, out_dtype=torch.float32, max_context_len=None):
    """Scatter each sequence's new token, then decode; returns the output tensor."""
    b = db.h
    slots = torch.from_numpy(new_token_slots(b)).cuda()
    pa.pa_reshape_and_cache(db.new_key, db.new_value, db.k_cache, db.v_cache, slots)
    out = torch.empty((b.num_seqs, b.num_heads, b.head_dim), dtype=out_dtype, device="cuda")
    mcl = b.max_context_len if max_context_len is None else max_context_len
    pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens, mcl,
                 b.scale, workspace=workspace)
    return out


def make_workspace(b, max_context_len=None):
    n = pa.pa_decode_workspace_size(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim,
                                    b.block_size, b.max_context_len if max_context_len is None
                                    else max_context_len)
    return torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")


def oracle_step(batch, nthreads=None):
    """Oracle: the same scatter, then fp64 attention. Returns (out, k_cache, v_cache)."""
    k = batch.k_cache.copy()
    v = batch.v_cache.copy()
    seq = np.arange(batch.num_seqs)
    slots = oracle.slot_mapping(batch.block_tables, seq, batch.new_pos, batch.block_size)
    oracle.reshape_and_cache(k, v, batch.new_key, batch.new_value, slots)
    out = oracle.paged_attention(batch.query, k, v, batch.block_tables, batch.context_lens,
                                 batch.scale, nthreads=nthreads)
    return out, k, v


def max_err(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape
    assert np.all(np.isfinite(g))
    return float(np.max(np.abs(g - want))) if g.size else 0.0
