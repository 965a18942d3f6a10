"""ORACLE -- TEST INFRASTRUCTURE ONLY. Slot ids, slot scatter and block copy.

* Slot id: "Paged Attention: Virtual Memory for the KV Cache", section
  "Finding a token: position, block, slot" -- slot = block number x block
  size + offset, with the block number read from the block table at the
  token's logical block (position // block size) and the offset
  position % block size ("What Does PagedAttention Actually Optimize?",
  section 17, write_kv).
* Scatter (reshape_and_cache): the key and value of each new token go into
  its slot, for every KV head ("PagedAttention, explained.", procedure step 4
  and the fused write kernels named under "Across GPUs"). A negative slot
  means "no token here" and is skipped (a convention the pages leave open).
* Copy (copy_blocks): copy-on-write duplicates a whole block before the
  writer touches it ("PagedAttention: KV cache virtual memory", section
  "Copy-on-write: when two requests share a prefix"; "How PagedAttention
  Eliminates KV-Cache Fragmentation", section "Advanced Memory Sharing and
  Copy-on-Write").

* Swap (swap_blocks): a preempted request's blocks are copied whole to CPU
  memory and back ("PagedAttention, explained.", procedure steps 7-8; "What
  Does PagedAttention Actually Optimize?", section 12): block dst of the
  destination pool becomes a copy of block src of the source pool. A pair
  naming a block outside its pool is skipped (the library's convention).

Arrays are numpy; the caches are [num_blocks, block_size, Hkv, D] and are
modified in place.
"""
from __future__ import annotations

import numpy as np


def slot_mapping(block_tables: np.ndarray, seq_index, positions, block_size: int) -> np.ndarray:
    """slot[i] = table[seq[i]][pos[i] // B] * B + pos[i] % B; pos < 0 gives -1."""
    out = np.empty(len(positions), dtype=np.int64)
    for i, (s, p) in enumerate(zip(seq_index, positions)):
        s, p = int(s), int(p)
        if p < 0:
            out[i] = -1
            continue
        logical = p // block_size
        offset = p % block_size
        out[i] = int(block_tables[s][logical]) * block_size + offset
    return out


def reshape_and_cache(k_cache: np.ndarray, v_cache: np.ndarray, key: np.ndarray,
                      value: np.ndarray, slots) -> None:
    """Write key[i], value[i] ([Hkv, D] each) into slot slots[i] of the caches."""
    B = k_cache.shape[1]
    for i, slot in enumerate(slots):
        slot = int(slot)
        if slot < 0:
            continue
        block, offset = slot // B, slot % B
        k_cache[block, offset] = key[i]
        v_cache[block, offset] = value[i]


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_mapping) -> None:
    """For each (src, dst) pair, block dst of both caches becomes a copy of src."""
    for src, dst in block_mapping:
        k_cache[int(dst)] = k_cache[int(src)]
        v_cache[int(dst)] = v_cache[int(src)]


def swap_blocks(dst_k: np.ndarray, dst_v: np.ndarray, src_k: np.ndarray, src_v: np.ndarray,
                block_mapping) -> None:
    """For each (src, dst) pair, block dst of (dst_k, dst_v) becomes a copy of
    block src of (src_k, src_v); pairs outside either pool are skipped."""
    for src, dst in block_mapping:
        src, dst = int(src), int(dst)
        if 0 <= src < src_k.shape[0] and 0 <= dst < dst_k.shape[0]:
            dst_k[dst] = src_k[src]
            dst_v[dst] = src_v[src]
