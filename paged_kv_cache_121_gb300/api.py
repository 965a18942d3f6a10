"""Python binding of libpa: one function per C entry point, same names.

Argument marshalling only -- shapes are read off the tensors, pointers and
the current CUDA stream are passed through, and a non-OK status raises
:class:`PAError`. Every computation runs in libpa's kernels (or, for the
block manager and slot map, in its host C++).
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np
import torch

from . import _lib

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_BLOCKS = 0, 1, 2, 3
PA_ERR_WORKSPACE, PA_ERR_TIMEOUT, PA_ERR_CUDA, PA_ERR_NOT_FOUND = 4, 5, 6, 7
PA_F32, PA_BF16, PA_F16 = 0, 1, 2


class PAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        text = _lib.load().pa_status_string(status).decode()
        super().__init__(f"{where}: {text} (status {status})")


def _check(status: int, where: str) -> None:
    if status != PA_OK:
        raise PAError(status, where)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PA_F32
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype == torch.float16:
        return PA_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libpa must be contiguous")
    return t.data_ptr()   # an int: ctypes converts it through the c_void_p argtype


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _cache_dims(k_cache: torch.Tensor) -> Tuple[int, int, int, int]:
    if k_cache.dim() != 4:
        raise ValueError("caches are [num_blocks, block_size, num_kv_heads, head_dim]")
    return tuple(int(x) for x in k_cache.shape)


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Write key[i], value[i] ([T, Hkv, D]) into slot slot_mapping[i] (int64) of the caches."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T = int(slot_mapping.numel())
    if T and tuple(key.shape) != (T, hkv, d):
        raise ValueError("key must be [num_tokens, num_kv_heads, head_dim]")
    _check(_lib.load().pa_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(slot_mapping), T, nb, bs, hkv, d, _dtype(k_cache),
                                           _stream(stream)), "pa_reshape_and_cache")


def pa_copy_blocks(k_cache, v_cache, block_mapping, stream=None) -> None:
    """For each (src, dst) row of block_mapping ([N, 2] int64), copy block src to dst."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    if block_mapping.dtype != torch.int64:
        raise TypeError("block_mapping must be int64")
    N = int(block_mapping.shape[0]) if block_mapping.numel() else 0
    _check(_lib.load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_mapping), N, nb, bs,
                                     hkv, d, _dtype(k_cache), _stream(stream)), "pa_copy_blocks")


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                             max_context_len) -> int:
    return int(_lib.load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                    block_size, max_context_len))


class DecodePlan(ctypes.Structure):
    """pa_decode_plan_t: how pa_decode runs a problem on the current device."""
    _fields_ = [("tensor_cores", ctypes.c_int), ("heads_per_cta", ctypes.c_int),
                ("num_splits", ctypes.c_int), ("partition_tokens", ctypes.c_int),
                ("cluster_merge", ctypes.c_int), ("kernel_launches", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("balanced", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


def pa_decode_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                   kv_dtype=PA_BF16, with_workspace=True) -> dict:
    """The plan pa_decode uses for this problem (host only; no launch)."""
    plan = DecodePlan()
    _check(_lib.load().pa_decode_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                     max_context_len, int(kv_dtype), int(bool(with_workspace)),
                                     ctypes.byref(plan)), "pa_decode_plan")
    return plan.as_dict()


def pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
              workspace=None, stream=None) -> None:
    """Paged decode attention into ``out`` [B, Hq, D] (float32, bfloat16 or float16).

    ``workspace`` is a uint8 tensor of at least :func:`pa_decode_workspace_size`
    bytes (its contents need no initialisation; calls sharing it must not
    overlap on the GPU), or None: then the tensor-core kernel merges a split of
    up to 8 partitions inside a thread-block cluster and trims a wider one to
    8, and the CUDA-core kernel does not split."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, dq = (int(x) for x in query.shape)
    ws_bytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    _check(_lib.load().pa_decode(_ptr(out), _dtype(out), _ptr(query), _dtype(query), _ptr(k_cache),
                                _ptr(v_cache), _dtype(k_cache), _ptr(block_tables),
                                _ptr(context_lens), B, hq, hkv, d, bs, int(block_tables.shape[1]),
                                nb, int(max_context_len), float(scale), _ptr(workspace), ws_bytes,
                                _stream(stream)), "pa_decode")


def pa_decode_append(out, query, new_key, new_value, k_cache, v_cache, block_tables, context_lens,
                     max_context_len, scale, workspace=None, stream=None) -> None:
    """One decode step: sequence b's new token (``new_key[b]``, ``new_value[b]``,
    [B, Hkv, D]) is written to position ``context_lens[b] - 1`` through its
    block table, then :func:`pa_decode` runs into ``out``."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, _ = (int(x) for x in query.shape)
    if tuple(new_key.shape) != (B, hkv, d) or tuple(new_value.shape) != (B, hkv, d):
        raise ValueError("new_key / new_value must be [num_seqs, num_kv_heads, head_dim]")
    ws_bytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    _check(_lib.load().pa_decode_append(_ptr(out), _dtype(out), _ptr(query), _dtype(query), _ptr(new_key),
                                       _ptr(new_value), _ptr(k_cache), _ptr(v_cache), _dtype(k_cache),
                                       _ptr(block_tables), _ptr(context_lens), B, hq, hkv, d, bs,
                                       int(block_tables.shape[1]), nb, int(max_context_len), float(scale),
                                       _ptr(workspace), ws_bytes, _stream(stream)), "pa_decode_append")


def pa_swap_blocks(dst_k, dst_v, src_k, src_v, block_mapping, stream=None) -> None:
    """Copy blocks block_mapping[i, 0] of (src_k, src_v) to blocks
    block_mapping[i, 1] of (dst_k, dst_v); either pool may be a pinned host
    tensor, the mapping a device or pinned host int64 tensor [n, 2]."""
    snb, bs, hkv, d = _cache_dims(src_k)
    dnb = int(dst_k.shape[0])
    _check(_lib.load().pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v), _ptr(block_mapping),
                                     int(block_mapping.shape[0]), snb, dnb, bs, hkv, d, _dtype(src_k),
                                     _stream(stream)), "pa_swap_blocks")


def pa_decode_shared_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                           max_context_len, shared_blocks) -> int:
    return int(_lib.load().pa_decode_shared_prefix_workspace_size(
        num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, shared_blocks))


def pa_decode_shared_prefix(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len,
                            shared_blocks, scale, workspace, stream=None) -> None:
    """Decode attention where the first ``shared_blocks`` entries of every
    block-table row are the same (full) physical blocks: they are read once
    for the whole batch. ``workspace``: a uint8 tensor of at least
    :func:`pa_decode_shared_prefix_workspace_size` bytes."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, _ = (int(x) for x in query.shape)
    ws_bytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    _check(_lib.load().pa_decode_shared_prefix(
        _ptr(out), _dtype(out), _ptr(query), _dtype(query), _ptr(k_cache), _ptr(v_cache), _dtype(k_cache),
        _ptr(block_tables), _ptr(context_lens), B, hq, hkv, d, bs, int(block_tables.shape[1]), nb,
        int(max_context_len), int(shared_blocks), float(scale), _ptr(workspace), ws_bytes, _stream(stream)),
        "pa_decode_shared_prefix")


def pa_decode_contiguous(out, query, k, v, context_lens, max_context_len, scale, workspace=None,
                         stream=None) -> None:
    """Decode attention over a contiguous cache ``k``, ``v`` [B, max_seq_len,
    Hkv, D] (bfloat16 or float16, no block table): the unpaged baseline. ``workspace``
    as for :func:`pa_decode`, sized with block_size 16."""
    B, L, hkv, d = (int(x) for x in k.shape)
    _, hq, _ = (int(x) for x in query.shape)
    ws_bytes = int(workspace.numel() * workspace.element_size()) if workspace is not None else 0
    _check(_lib.load().pa_decode_contiguous(_ptr(out), _dtype(out), _ptr(query), _dtype(query), _ptr(k),
                                           _ptr(v), _dtype(k), _ptr(context_lens), B, hq, hkv, d, L,
                                           int(max_context_len), float(scale), _ptr(workspace), ws_bytes,
                                           _stream(stream)), "pa_decode_contiguous")


def pa_decode_static_scratch(out, query, k_cache, v_cache, block_tables, context_lens, max_context_len,
                             scale, stream=None) -> None:
    """pa_decode without a workspace argument, for callers that cannot
    allocate device memory: a split of up to 8 partitions is merged inside a
    thread-block cluster, a wider one through the library's own fixed
    scratch (calls must not overlap on the GPU)."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, _ = (int(x) for x in query.shape)
    _check(_lib.load().pa_decode_static_scratch(
        _ptr(out), _dtype(out), _ptr(query), _dtype(query), _ptr(k_cache), _ptr(v_cache),
        _dtype(k_cache), _ptr(block_tables), _ptr(context_lens), B, hq, hkv, d, bs,
        int(block_tables.shape[1]), nb, int(max_context_len), float(scale), _stream(stream)),
        "pa_decode_static_scratch")


def pa_decode_splitk(tmp_out, max_logits, exp_sums, partition_size, query, k_cache, v_cache,
                     block_tables, context_lens, max_context_len, scale, stream=None) -> None:
    """Per-partition attention: tmp_out [B, Hq, P, D], max_logits / exp_sums [B, Hq, P] (float32)."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, _ = (int(x) for x in query.shape)
    _check(_lib.load().pa_decode_splitk(_ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums),
                                       int(partition_size), _ptr(query), _dtype(query),
                                       _ptr(k_cache), _ptr(v_cache), _dtype(k_cache),
                                       _ptr(block_tables), _ptr(context_lens), B, hq, hkv, d, bs,
                                       int(block_tables.shape[1]), nb, int(max_context_len),
                                       float(scale), _stream(stream)), "pa_decode_splitk")


def pa_lse_merge(out, tmp_out, max_logits, exp_sums, context_lens, partition_size, stream=None) -> None:
    """Log-sum-exp merge of pa_decode_splitk's partitions into ``out`` [B, Hq, D]."""
    B, hq, P, d = (int(x) for x in tmp_out.shape)
    _check(_lib.load().pa_lse_merge(_ptr(out), _dtype(out), _ptr(tmp_out), _ptr(max_logits),
                                   _ptr(exp_sums), _ptr(context_lens), B, hq, d, P,
                                   int(partition_size), _stream(stream)), "pa_lse_merge")


def pa_device_status(clear: bool = True, stream=None) -> int:
    """The device status word (0, or PA_ERR_TIMEOUT after a kernel gave up waiting)."""
    v = ctypes.c_int(0)
    _check(_lib.load().pa_device_status(ctypes.byref(v), int(clear), _stream(stream)), "pa_device_status")
    return v.value


def pa_check_wait_timeout(timeout_us: int = 1000, stream=None) -> None:
    """Run the failure-detection check: one CTA's bounded wait on a stage no
    copy fills runs out after ``timeout_us`` and records PA_ERR_TIMEOUT in the
    device status word (read it with :func:`pa_device_status`)."""
    _check(_lib.load().pa_check_wait_timeout(int(timeout_us), _stream(stream)), "pa_check_wait_timeout")


def pa_compute_slot_mapping(block_tables: np.ndarray, seq_index, positions, block_size: int) -> np.ndarray:
    """Host slot map: table[seq][pos // B] * B + pos % B (pos < 0 -> -1)."""
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    seq = np.ascontiguousarray(seq_index, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty(pos.shape[0], dtype=np.int64)
    _check(_lib.load().pa_compute_slot_mapping(
        out.ctypes.data_as(_lib.P_I64), tables.ctypes.data_as(_lib.P_I32), tables.shape[0],
        tables.shape[1], seq.ctypes.data_as(_lib.P_I32), pos.ctypes.data_as(_lib.P_I32),
        pos.shape[0], int(block_size)), "pa_compute_slot_mapping")
    return out


class BlockManager:
    """Handle on the host block manager (pa_bm_*)."""

    def __init__(self, num_blocks: int, block_size: int, reserve_null_block: bool = True,
                 free_order=None):
        self._lib = _lib.load()
        h = ctypes.c_void_p()
        if free_order is None:
            st = self._lib.pa_bm_create(num_blocks, block_size, int(reserve_null_block), ctypes.byref(h))
        else:
            arr = np.ascontiguousarray(free_order, dtype=np.int32)
            st = self._lib.pa_bm_create_with_free_list(num_blocks, block_size,
                                                       arr.ctypes.data_as(_lib.P_I32), arr.size,
                                                       ctypes.byref(h))
        _check(st, "pa_bm_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def allocate(self, seq: int, num_tokens: int) -> None:
        _check(self._lib.pa_bm_allocate(self._h, seq, num_tokens), "pa_bm_allocate")

    def append_slot(self, seq: int) -> Tuple[int, int, int]:
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pa_bm_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                           ctypes.byref(dst)), "pa_bm_append_slot")
        return slot.value, src.value, dst.value

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_bm_fork(self._h, parent, child), "pa_bm_fork")

    def free(self, seq: int) -> None:
        _check(self._lib.pa_bm_free(self._h, seq), "pa_bm_free")

    def _list(self, fn, *args):
        n = ctypes.c_int(0)
        fn(self._h, *args, None, 0, ctypes.byref(n))
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check(fn(self._h, *args, buf, n.value, ctypes.byref(n)), fn.__name__)
        return [int(buf[i]) for i in range(n.value)]

    def block_table(self, seq: int):
        return self._list(self._lib.pa_bm_block_table, seq)

    def free_list(self):
        return self._list(self._lib.pa_bm_free_list)

    def num_tokens(self, seq: int) -> int:
        n = ctypes.c_int()
        _check(self._lib.pa_bm_num_tokens(self._h, seq, ctypes.byref(n)), "pa_bm_num_tokens")
        return n.value

    def refcount(self, block: int) -> int:
        n = ctypes.c_int()
        _check(self._lib.pa_bm_refcount(self._h, block, ctypes.byref(n)), "pa_bm_refcount")
        return n.value

    def stats(self) -> dict:
        s = _lib.PaBmStats()
        _check(self._lib.pa_bm_stats(self._h, ctypes.byref(s)), "pa_bm_stats")
        return {name: int(getattr(s, name)) for name, _ in _lib.PaBmStats._fields_}

    # -- swapping to a CPU pool -------------------------------------------
    def enable_swap(self, num_host_blocks: int) -> None:
        _check(self._lib.pa_bm_enable_swap(self._h, num_host_blocks), "pa_bm_enable_swap")

    def _swap(self, fn, seqs) -> np.ndarray:
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        cap = int(sum(len(self.block_table(int(s))) for s in ids)) if ids.size else 0
        out = np.zeros((max(cap, 1), 2), dtype=np.int64)
        n = ctypes.c_int(0)
        _check(fn(self._h, ids.ctypes.data_as(_lib.P_I64), ids.size, out.ctypes.data_as(_lib.P_I64), cap,
                  ctypes.byref(n)), fn.__name__)
        return out[: n.value].copy()

    def swap_out(self, seqs) -> np.ndarray:
        """Move a group of sequences to the CPU pool; returns [n, 2] (GPU id, CPU id) pairs."""
        return self._swap(self._lib.pa_bm_swap_out, seqs)

    def swap_in(self, seqs) -> np.ndarray:
        """Bring a swapped-out group back; returns [n, 2] (CPU id, GPU id) pairs."""
        return self._swap(self._lib.pa_bm_swap_in, seqs)

    def is_swapped(self, seq: int) -> bool:
        v = ctypes.c_int(0)
        _check(self._lib.pa_bm_is_swapped(self._h, seq, ctypes.byref(v)), "pa_bm_is_swapped")
        return bool(v.value)

    def swap_stats(self) -> dict:
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pa_bm_swap_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "pa_bm_swap_stats")
        return {"host_blocks": a.value, "free_host_blocks": b.value, "swapped_seqs": c.value}
