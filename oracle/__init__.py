"""ORACLE -- TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 CPU statement of the paged-KV-cache hot path, written from
the source pages and independent of the CUDA path (no shared code, headers,
tables or helpers; neither imports the other). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline may import it.

Contents:
  * paged decode attention, whole-context and per-partition, and the
    log-sum-exp merge (C, ``paged_attention.c``, via ctypes); caches and
    queries are fp32, bf16 (as uint16 bits) or fp16, all widened exactly;
  * the slot scatter (reshape_and_cache), the block copy (copy_blocks) and the
    slot-id formula (numpy, ``cache_ops.py``);
  * a list-based model of the block manager (``block_manager_model.py``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle
from .cache_ops import copy_blocks, reshape_and_cache, slot_mapping, swap_blocks  # noqa: F401
from .block_manager_model import BlockManagerModel, OutOfBlocks  # noqa: F401

_lib = None


def load_library(path: str):
    """Load an oracle shared library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    i32p = ctypes.POINTER(ctypes.c_int32)
    ci, cd = ctypes.c_int, ctypes.c_double
    lib.oracle_paged_attention_partitions.argtypes = [
        dp, dp, dp, dp, vp, vp, ci, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, cd, ci, ci, ci]
    lib.oracle_paged_attention_partitions.restype = ci
    lib.oracle_paged_attention.argtypes = [
        dp, dp, vp, vp, ci, i32p, ci, i32p, ci, ci, ci, ci, ci, ci, cd, ci]
    lib.oracle_paged_attention.restype = ci
    lib.oracle_lse_merge.argtypes = [dp, dp, dp, dp, ci, ci, ci]
    lib.oracle_lse_merge.restype = ci
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    if _lib is None:
        _lib = load_library(build_oracle())
    return _lib


def _widen_query(query: np.ndarray, bf16: bool) -> np.ndarray:
    if bf16:
        bits = np.ascontiguousarray(query, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.ascontiguousarray(query, dtype=np.float64)


def _cache_args(k_cache: np.ndarray, v_cache: np.ndarray):
    if v_cache.dtype != k_cache.dtype or v_cache.shape != k_cache.shape:
        raise TypeError("k_cache and v_cache must match")
    if k_cache.dtype == np.uint16:
        bf16 = True
    elif k_cache.dtype == np.float32:
        bf16 = False
    elif k_cache.dtype == np.float16:
        # every fp16 value is an fp32 value: widening is exact
        return k_cache.astype(np.float32), v_cache.astype(np.float32), False
    else:
        raise TypeError("cache must be float32, float16 or uint16 (bf16 bits)")
    return np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache), bf16


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def default_threads() -> int:
    return os.cpu_count() or 1


def paged_attention(query, k_cache, v_cache, block_tables, context_lens, scale,
                    query_bf16=None, nthreads=None, lib=None) -> np.ndarray:
    """Decode attention through the block table; returns float64 [B, Hq, D]."""
    k, v, bf16 = _cache_args(k_cache, v_cache)
    qb = (query.dtype == np.uint16) if query_bf16 is None else query_bf16
    q = _widen_query(query, qb)
    B, Hq, D = q.shape
    nb, bs, hkv, d2 = k.shape
    assert d2 == D
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load(lib).oracle_paged_attention(
        _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_double), k.ctypes.data, v.ctypes.data,
        int(bf16), _ptr(tables, ctypes.c_int32), tables.shape[1], _ptr(lens, ctypes.c_int32),
        B, Hq, hkv, D, bs, nb, float(scale), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_paged_attention rejected its arguments")
    return out


def paged_attention_partitions(query, k_cache, v_cache, block_tables, context_lens, scale,
                               partition_size, num_partitions, query_bf16=None, nthreads=None,
                               lib=None):
    """Per-partition attention: (out [B,Hq,P,D], max [B,Hq,P], sum [B,Hq,P]) in float64."""
    k, v, bf16 = _cache_args(k_cache, v_cache)
    qb = (query.dtype == np.uint16) if query_bf16 is None else query_bf16
    q = _widen_query(query, qb)
    B, Hq, D = q.shape
    nb, bs, hkv, _ = k.shape
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    P = int(num_partitions)
    out = np.empty((B, Hq, P, D), dtype=np.float64)
    mx = np.empty((B, Hq, P), dtype=np.float64)
    sm = np.empty((B, Hq, P), dtype=np.float64)
    rc = _load(lib).oracle_paged_attention_partitions(
        _ptr(out, ctypes.c_double), _ptr(mx, ctypes.c_double), _ptr(sm, ctypes.c_double),
        _ptr(q, ctypes.c_double), k.ctypes.data, v.ctypes.data, int(bf16),
        _ptr(tables, ctypes.c_int32), tables.shape[1], _ptr(lens, ctypes.c_int32),
        B, Hq, hkv, D, bs, nb, float(scale), int(partition_size), P,
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_paged_attention_partitions rejected its arguments")
    return out, mx, sm


def lse_merge(part_out, part_max, part_sum, lib=None) -> np.ndarray:
    """Merge partitions by log-sum-exp; returns float64 [..., D]."""
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    mx = np.ascontiguousarray(part_max, dtype=np.float64)
    sm = np.ascontiguousarray(part_sum, dtype=np.float64)
    lead = po.shape[:-2]
    P, D = po.shape[-2:]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (D,), dtype=np.float64)
    rc = _load(lib).oracle_lse_merge(_ptr(out, ctypes.c_double), _ptr(po, ctypes.c_double),
                                  _ptr(mx, ctypes.c_double), _ptr(sm, ctypes.c_double),
                                  rows, P, D)
    if rc != 0:
        raise ValueError("oracle_lse_merge rejected its arguments")
    return out
