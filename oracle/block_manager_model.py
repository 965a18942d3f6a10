"""ORACLE -- TEST INFRASTRUCTURE ONLY. A list-based model of the KV block manager.

What it follows:
  * "Paged Attention: Virtual Memory for the KV Cache", sections "Paging:
    blocks handed out as tokens arrive" (free list; cdiv(num_tokens,
    block_size) blocks for a prompt; one more block each time the last one
    fills; blocks return to the free list when the request ends) and "Inside
    vLLM: the block pool" (block 0 is never handed out; allocation takes from
    the front of the free queue; a block whose count drops to zero and whose
    contents are not reusable goes to the front, so it is reused first).
  * "PagedAttention, explained.", procedure steps 1-4 and 6 (free list, block
    table, prefill allocation, decode fills the last block, reference counts
    and copy-on-write when writing into a block whose count is above one).
  * "PagedAttention: KV cache virtual memory", section "Copy-on-write": the
    writer gets a clone, the original's count drops by one, only the
    writer's table changes.

  * "PagedAttention, explained.", procedure steps 7-8 and "What Does
    PagedAttention Actually Optimize?", section 12 (swapping): when blocks
    run out, a request's blocks are evicted all at once -- sequences that
    share blocks together -- copied to CPU memory, and copied back later.

Readings where the pages are open: freed blocks go to the queue front in
block-table order; a fork copies the parent's table and token count and adds
one reference to each block; the free queue starts in ascending id order
unless an explicit order is given. Swapping: the CPU pool is a second free
queue (ascending ids, freed to the front); a swapped group must hold every
reference to its blocks; each distinct block, in order of first appearance
across the group's tables, takes the next block of the other pool, and the
blocks it leaves go to the front of their queue in that order; a swapped-out
sequence cannot grow or fork until it is swapped back in.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class OutOfBlocks(RuntimeError):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int, reserve_null_block: bool = True,
                 free_order: Optional[Sequence[int]] = None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.reserve_null_block = reserve_null_block
        if free_order is None:
            first = 1 if reserve_null_block else 0
            self.free: List[int] = list(range(first, num_blocks))
        else:
            self.free = [int(b) for b in free_order]
        self.refcount: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.tokens: Dict[int, int] = {}
        self.cow_copies = 0
        self.host_free: Optional[List[int]] = None   # CPU pool, once swapping is enabled
        self.host_ref: List[int] = []
        self.swapped: set = set()

    # -- helpers ---------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free block")
        b = self.free.pop(0)
        self.refcount[b] = 1
        return b

    # -- operations ------------------------------------------------------
    def allocate(self, seq: int, num_tokens: int) -> List[int]:
        if seq in self.tables:
            raise KeyError("sequence exists")
        if num_tokens < 0:
            raise ValueError("negative token count")
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks("not enough free blocks")
        self.tables[seq] = [self._take() for _ in range(need)]
        self.tokens[seq] = num_tokens
        return list(self.tables[seq])

    def append_slot(self, seq: int) -> Tuple[int, int, int]:
        """Make room for one more token; returns (slot, cow_src, cow_dst)."""
        if seq in self.swapped:
            raise ValueError("sequence is swapped out")
        table = self.tables[seq]
        pos = self.tokens[seq]
        offset = pos % self.block_size
        src = dst = -1
        if offset == 0 and len(table) * self.block_size <= pos:
            table.append(self._take())
        else:
            last = table[pos // self.block_size]
            if self.refcount[last] > 1:
                new = self._take()
                self.refcount[last] -= 1
                table[pos // self.block_size] = new
                src, dst = last, new
                self.cow_copies += 1
        slot = table[pos // self.block_size] * self.block_size + offset
        self.tokens[seq] = pos + 1
        return slot, src, dst

    def fork(self, parent: int, child: int) -> None:
        table = self.tables[parent]
        if child in self.tables or parent in self.swapped:
            raise ValueError("child exists or parent swapped out")
        for b in table:
            self.refcount[b] += 1
        self.tables[child] = list(table)
        self.tokens[child] = self.tokens[parent]

    def free_seq(self, seq: int) -> None:
        table = self.tables.pop(seq)
        del self.tokens[seq]
        ref, free = (self.host_ref, self.host_free) if seq in self.swapped else (self.refcount, self.free)
        self.swapped.discard(seq)
        released = []
        for b in table:
            ref[b] -= 1
            if ref[b] == 0:
                released.append(b)
        free[0:0] = released

    # -- swapping ----------------------------------------------------------
    def enable_swap(self, num_host_blocks: int) -> None:
        if self.host_free is not None or num_host_blocks <= 0:
            raise ValueError("swap already enabled or empty pool")
        self.host_free = list(range(num_host_blocks))
        self.host_ref = [0] * num_host_blocks

    def _swap(self, seqs, out: bool) -> List[Tuple[int, int]]:
        if self.host_free is None:
            raise ValueError("swap not enabled")
        seqs = [int(x) for x in seqs]
        for q in seqs:
            if q not in self.tables:
                raise KeyError("unknown sequence")
        if len(set(seqs)) != len(seqs) or any((q in self.swapped) == out for q in seqs):
            raise ValueError("duplicate sequence or wrong swap state")
        order: List[int] = []
        refs: Dict[int, int] = {}
        for q in seqs:
            for b in self.tables[q]:
                if b not in refs:
                    refs[b] = 0
                    order.append(b)
                refs[b] += 1
        src_ref, dst_ref = (self.refcount, self.host_ref) if out else (self.host_ref, self.refcount)
        src_free, dst_free = (self.free, self.host_free) if out else (self.host_free, self.free)
        if any(src_ref[b] != refs[b] for b in order):
            raise ValueError("a block is shared with a sequence outside the group")
        if len(order) > len(dst_free):
            raise OutOfBlocks("destination pool too small")
        moved = {}
        for b in order:
            nb = dst_free.pop(0)
            dst_ref[nb] = src_ref[b]
            src_ref[b] = 0
            moved[b] = nb
        src_free[0:0] = order
        for q in seqs:
            self.tables[q] = [moved[b] for b in self.tables[q]]
            if out:
                self.swapped.add(q)
            else:
                self.swapped.discard(q)
        return [(b, moved[b]) for b in order]

    def swap_out(self, seqs) -> List[Tuple[int, int]]:
        """Evict a group to the CPU pool; returns (GPU id, CPU id) pairs."""
        return self._swap(seqs, True)

    def swap_in(self, seqs) -> List[Tuple[int, int]]:
        """Bring a group back; returns (CPU id, GPU id) pairs."""
        return self._swap(seqs, False)

    # -- queries ---------------------------------------------------------
    def block_table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def num_tokens(self, seq: int) -> int:
        return self.tokens[seq]

    def stats(self) -> dict:
        usable = self.num_blocks - (1 if self.reserve_null_block else 0)
        used = sum(1 for r in self.refcount if r > 0)
        shared = sum(1 for r in self.refcount if r > 1)
        logical = sum(len(t) for t in self.tables.values())
        tokens = sum(self.tokens.values())
        return {
            "num_blocks": usable,
            "free_blocks": len(self.free),
            "used_blocks": used,
            "shared_blocks": shared,
            "num_seqs": len(self.tables),
            "logical_blocks": logical,
            "num_tokens": tokens,
            "waste_slots": logical * self.block_size - tokens,
            "cow_copies": self.cow_copies,
        }
