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

Readings where the pages are open: freed blocks go to the queue front in
block-table order; a fork copies the parent's table and token count and adds
one reference to each block; the free queue starts in ascending id order
unless an explicit order is given.
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
        if child in self.tables:
            raise KeyError("child exists")
        table = self.tables[parent]
        for b in table:
            self.refcount[b] += 1
        self.tables[child] = list(table)
        self.tokens[child] = self.tokens[parent]

    def free_seq(self, seq: int) -> None:
        table = self.tables.pop(seq)
        del self.tokens[seq]
        released = []
        for b in table:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                released.append(b)
        self.free[0:0] = released

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
