"""Seeded synthetic inputs for paged decode attention.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests. It only draws random numbers, rounds the draws to bf16, and
places each sequence's logical blocks onto physical block ids; it computes no
attention, no slot ids and no copies (that arithmetic lives, independently, in
the kernels and in the oracle).

Recipe (fixed seeds, numpy PCG64 ``default_rng``):
  * seed 121: K/V/query values, N(0, 1) drawn in fp32, then rounded to bf16
    (or, for fp16 batches, to fp16) with round-to-nearest-even (the toy case
    stays fp32);
  * seed 122: physical block placement, ``rng.permutation(num_blocks)`` taken
    in order, one id per logical block, sequence after sequence;
  * seed 123: context lengths and shared-prefix suffix lengths.

Workload shapes follow the pages: the 25/47/12-token toy of "PagedAttention:
KV cache virtual memory" (section "A small worked example"); the Qwen3-8B
layer of "Paged Attention: Virtual Memory for the KV Cache" (36 layers x 8 KV
heads x 128 dims bf16, 16 requests of 4,100 + 64 tokens, 38,348 blocks of 16,
section "Measured: the same prompt, sixteen at a time"), plus a Llama-style
GQA batch, a shared-prefix copy-on-write batch and a long-context batch.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

SEED_VALUES = 121
SEED_BLOCKS = 122
SEED_LENGTHS = 123


# --------------------------------------------------------------------------
# bf16 helpers (storage format only: bf16 values are carried as uint16 bits)
# --------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).copy()
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    b += np.uint32(0x7FFF)
    b += lsb
    b >>= np.uint32(16)
    return b.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to fp32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng: np.random.Generator, shape, bf16: bool, f16: bool = False) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if bf16:
        return bf16_round(x)
    return x.astype(np.float16) if f16 else x


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


# --------------------------------------------------------------------------
# A decode batch: a block pool, per-sequence block tables, one query per head
# --------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeBatch:
    """One decode step's inputs.

    Arrays (row-major, numpy):
      query        [B, Hq, D]                 float32, float16, or uint16 bf16 bits
      k_cache      [num_blocks, BS, Hkv, D]   float32, float16, or uint16 bf16 bits
      v_cache      same as k_cache
      block_tables [B, max_blocks] int32, entries past a sequence's blocks = 0
      context_lens [B] int32 (the number of tokens attended, new token included)
      new_key      [B, Hkv, D] the token written this step (same dtype as cache)
      new_value    [B, Hkv, D]
      new_pos      [B] int32 position of that token (= context_len - 1)
    """
    name: str
    query: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    new_key: np.ndarray
    new_value: np.ndarray
    new_pos: np.ndarray
    block_size: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    bf16: bool
    f16: bool = False

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def elem_bytes(self) -> int:
        return 2 if self.bf16 or self.f16 else 4


def place_blocks(context_lens: np.ndarray, block_size: int, num_blocks: int,
                 max_blocks: Optional[int] = None, seed: int = SEED_BLOCKS,
                 exclude_zero: bool = False) -> np.ndarray:
    """Block tables whose physical ids are a seeded random permutation of the pool."""
    lens = np.asarray(context_lens, dtype=np.int64)
    need = [cdiv(int(n), block_size) for n in lens]
    if max_blocks is None:
        max_blocks = max(1, max(need) if need else 1)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_blocks).astype(np.int32)
    if exclude_zero:
        perm = perm[perm != 0]
    if sum(need) > perm.size:
        raise ValueError("pool too small for the requested lengths")
    tables = np.zeros((lens.size, max_blocks), dtype=np.int32)
    pos = 0
    for i, n in enumerate(need):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    return tables


def make_batch(name: str, context_lens, num_heads: int, num_kv_heads: int, head_dim: int,
               block_size: int, num_blocks: int, bf16: bool, max_blocks: Optional[int] = None,
               seed_values: int = SEED_VALUES, seed_blocks: int = SEED_BLOCKS,
               fill_unused: bool = False, f16: bool = False) -> DecodeBatch:
    """Draw a decode batch.

    Every slot of every block a sequence owns gets an N(0,1) draw, the tail
    slots of its last block included (so a kernel that forgets to mask them
    gives a wrong answer). Blocks nobody owns stay zero unless ``fill_unused``.
    ``f16`` (with ``bf16`` False): the draws are rounded to fp16 instead.
    """
    lens = np.asarray(context_lens, dtype=np.int32)
    B = lens.size
    tables = place_blocks(lens, block_size, num_blocks, max_blocks, seed_blocks)
    rng = np.random.default_rng(seed_values)
    f16 = f16 and not bf16
    dt = np.uint16 if bf16 else np.float16 if f16 else np.float32
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_cache = np.zeros(shape, dtype=dt)
    v_cache = np.zeros(shape, dtype=dt)
    used = [tables[i, :cdiv(int(n), block_size)] for i, n in enumerate(lens)]
    used = np.concatenate(used) if used else np.zeros(0, np.int32)
    if fill_unused:
        k_cache[...] = _normal(rng, shape, bf16, f16)
        v_cache[...] = _normal(rng, shape, bf16, f16)
    elif used.size:
        k_cache[used] = _normal(rng, (used.size,) + shape[1:], bf16, f16)
        v_cache[used] = _normal(rng, (used.size,) + shape[1:], bf16, f16)
    query = _normal(rng, (B, num_heads, head_dim), bf16, f16)
    new_key = _normal(rng, (B, num_kv_heads, head_dim), bf16, f16)
    new_value = _normal(rng, (B, num_kv_heads, head_dim), bf16, f16)
    return DecodeBatch(name=name, query=query, k_cache=k_cache, v_cache=v_cache,
                       block_tables=tables, context_lens=lens, new_key=new_key,
                       new_value=new_value, new_pos=np.maximum(lens - 1, 0).astype(np.int32),
                       block_size=block_size, num_heads=num_heads, num_kv_heads=num_kv_heads,
                       head_dim=head_dim, scale=1.0 / math.sqrt(head_dim), bf16=bf16, f16=f16)


def shared_prefix_batch(name: str, shared_blocks: int, suffix_lens, num_heads: int, num_kv_heads: int,
                        head_dim: int, block_size: int, spare_blocks: int = 7,
                        seed_values: int = SEED_VALUES, seed_blocks: int = SEED_BLOCKS,
                        f16: bool = False) -> DecodeBatch:
    """A bf16 (``f16``: fp16) decode batch whose sequences share their first ``shared_blocks``
    (full) blocks: every table row starts with the same physical ids, then
    each sequence's private blocks for ``suffix_lens[b]`` more tokens. Ids
    are a seeded permutation of a pool with ``spare_blocks`` unused blocks."""
    suffix = np.asarray(suffix_lens, dtype=np.int64)
    B = suffix.size
    lens = (shared_blocks * block_size + suffix).astype(np.int32)
    need_priv = [cdiv(int(n), block_size) - shared_blocks for n in lens]
    num_blocks = shared_blocks + sum(need_priv) + spare_blocks
    max_blocks = max(1, max(cdiv(int(n), block_size) for n in lens))
    perm = np.random.default_rng(seed_blocks).permutation(num_blocks).astype(np.int32)
    tables = np.zeros((B, max_blocks), dtype=np.int32)
    tables[:, :shared_blocks] = perm[:shared_blocks]
    pos = shared_blocks
    for b, n in enumerate(need_priv):
        tables[b, shared_blocks:shared_blocks + n] = perm[pos:pos + n]
        pos += n
    rng = np.random.default_rng(seed_values)
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_cache = np.zeros(shape, dtype=np.float16 if f16 else np.uint16)
    v_cache = np.zeros_like(k_cache)
    used = perm[:pos]
    k_cache[used] = _normal(rng, (used.size,) + shape[1:], not f16, f16)
    v_cache[used] = _normal(rng, (used.size,) + shape[1:], not f16, f16)
    query = _normal(rng, (B, num_heads, head_dim), not f16, f16)
    new_key = _normal(rng, (B, num_kv_heads, head_dim), not f16, f16)
    new_value = _normal(rng, (B, num_kv_heads, head_dim), not f16, f16)
    return DecodeBatch(name=name, query=query, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
                       context_lens=lens, new_key=new_key, new_value=new_value,
                       new_pos=np.maximum(lens - 1, 0).astype(np.int32), block_size=block_size,
                       num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                       scale=1.0 / math.sqrt(head_dim), bf16=not f16, f16=f16)


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------
TOY_LENS = (25, 47, 12)


def toy() -> DecodeBatch:
    """3 sequences of 25/47/12 tokens, blocks of 16 from a 64-block pool, fp32,
    Hq = Hkv = 4, D = 64, plus one new token per sequence."""
    return make_batch("toy", TOY_LENS, 4, 4, 64, 16, 64, bf16=False)


def gqa_lengths(num_seqs: int = 64, lo: int = 512, hi: int = 4096, seed: int = SEED_LENGTHS) -> np.ndarray:
    return np.random.default_rng(seed).integers(lo, hi + 1, size=num_seqs).astype(np.int32)


def gqa(num_seqs: int = 64, num_blocks: int = 20000, block_size: int = 16) -> DecodeBatch:
    """Llama-style GQA batch: lengths U[512, 4096], Hq 32, Hkv 8, D 128, blocks of 16."""
    return make_batch("gqa", gqa_lengths(num_seqs), 32, 8, 128, block_size, num_blocks, bf16=True)


GQA_UNIFORM_TOKENS = 2304    # the mean of U[512, 4096]: the same KV bytes as the ragged batch


def gqa_uniform(num_seqs: int = 64, num_blocks: int = 20000, block_size: int = 16) -> DecodeBatch:
    """The GQA batch with every length at the mean of U[512, 4096] (2,304
    tokens): the uniform counterpart of the ragged batch."""
    lens = np.full(num_seqs, GQA_UNIFORM_TOKENS, dtype=np.int32)
    return make_batch("gqa_uniform", lens, 32, 8, 128, block_size, num_blocks, bf16=True)


QWEN3_TOKENS = 4164          # 4,100-token prompt + 64 generated
QWEN3_POOL_BLOCKS = 38348    # 613,568 cache tokens / 16


def qwen3(num_seqs: int = 16, copies: int = 1, block_size: int = 16) -> DecodeBatch:
    """Qwen3-8B-shaped layer: ``num_seqs * copies`` sequences of 4,164 tokens,
    Hq 32, Hkv 8, D 128, bf16, blocks of 16 scattered over a 38,348-block pool.
    ``copies`` > 1 draws several disjoint batches in one pool (consecutive
    timed steps then read disjoint memory). Another ``block_size`` keeps the
    pool at 613,568 tokens."""
    lens = np.full(num_seqs * copies, QWEN3_TOKENS, dtype=np.int32)
    return make_batch("qwen3", lens, 32, 8, 128, block_size, QWEN3_POOL_BLOCKS * 16 // block_size,
                      bf16=True)


LONG_TOKENS = 32768
LONG_POOL_TOKENS = 9000 * 16   # the pool holds 144,000 tokens at any block size


def long_context(block_size: int = 16, num_seqs: int = 4, copies: int = 1) -> DecodeBatch:
    """4 sequences of 32,768 tokens, Hq 64, Hkv 8, D 128, bf16, pool of
    144,000 tokens (9,000 blocks at 16). ``copies`` > 1 draws several disjoint
    batches, each with its own 144,000-token share of the pool."""
    lens = np.full(num_seqs * copies, LONG_TOKENS, dtype=np.int32)
    return make_batch("long", lens, 64, 8, 128, block_size,
                      copies * LONG_POOL_TOKENS // block_size, bf16=True)


@dataclasses.dataclass
class ContiguousBatch:
    """One decode step's inputs over a contiguous (unpaged) cache: each
    sequence owns ``max_seq_len`` consecutive rows, as under a per-request
    maximum-length reservation.

      query        [B, Hq, D]              uint16 bf16 bits (float16 when not bf16)
      k, v         [B, max_seq_len, Hkv, D] uint16 bf16 bits (or float16); rows at or past a
                   sequence's length hold zeros, or NaN with ``tail_nan``
      context_lens [B] int32
      new_key, new_value [B, Hkv, D]; new_pos [B] (= context_len - 1)
    """
    name: str
    query: np.ndarray
    k: np.ndarray
    v: np.ndarray
    context_lens: np.ndarray
    new_key: np.ndarray
    new_value: np.ndarray
    new_pos: np.ndarray
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    bf16: bool = True

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_seq_len(self) -> int:
        return int(self.k.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    @property
    def elem_bytes(self) -> int:
        return 2


BF16_NAN_BITS = 0x7FC0


def contiguous(name: str, context_lens, num_heads: int, num_kv_heads: int, head_dim: int,
               max_seq_len: int, tail_nan: bool = False, seed_values: int = SEED_VALUES,
               f16: bool = False) -> ContiguousBatch:
    """Draw a bf16 (``f16``: fp16) decode batch in the contiguous layout
    (N(0,1) rows for each sequence's tokens, seeded like ``make_batch``)."""
    lens = np.asarray(context_lens, dtype=np.int32)
    B = lens.size
    if B and int(lens.max()) > max_seq_len:
        raise ValueError("a length exceeds max_seq_len")
    rng = np.random.default_rng(seed_values)
    shape = (B, max_seq_len, num_kv_heads, head_dim)
    if f16:
        dt, fill = np.float16, (np.float16(np.nan) if tail_nan else np.float16(0))
    else:
        dt, fill = np.uint16, (np.uint16(BF16_NAN_BITS) if tail_nan else np.uint16(0))
    k = np.full(shape, fill, dtype=dt)
    v = np.full(shape, fill, dtype=dt)
    for b in range(B):
        n = int(lens[b])
        k[b, :n] = _normal(rng, (n, num_kv_heads, head_dim), not f16, f16)
        v[b, :n] = _normal(rng, (n, num_kv_heads, head_dim), not f16, f16)
    query = _normal(rng, (B, num_heads, head_dim), not f16, f16)
    new_key = _normal(rng, (B, num_kv_heads, head_dim), not f16, f16)
    new_value = _normal(rng, (B, num_kv_heads, head_dim), not f16, f16)
    return ContiguousBatch(name=name, query=query, k=k, v=v, context_lens=lens, new_key=new_key,
                           new_value=new_value, new_pos=np.maximum(lens - 1, 0).astype(np.int32),
                           num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                           scale=1.0 / math.sqrt(head_dim), bf16=not f16)


@dataclasses.dataclass
class SharedPrefixCase:
    """Shared-prefix copy-on-write workload (values only; the block manager
    under test decides where blocks go)."""
    prefix_len: int
    suffix_lens: np.ndarray      # [S] int32
    block_size: int
    num_blocks: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    prefix_key: np.ndarray       # [prefix_len, Hkv, D] bf16 bits
    prefix_value: np.ndarray
    suffix_key: List[np.ndarray]     # per sequence [suffix_len + 1, Hkv, D] (suffix + decode token)
    suffix_value: List[np.ndarray]
    query: np.ndarray            # [S, Hq, D]
    scale: float


def shared_prefix(num_seqs: int = 64, prefix_len: int = 2048, max_suffix: int = 256,
                  block_size: int = 32, num_blocks: int = 8192, num_heads: int = 32,
                  num_kv_heads: int = 8, head_dim: int = 128) -> SharedPrefixCase:
    """64 sequences sharing one prefix, divergent suffixes U[0, 256] tokens,
    then one decode token each. ``prefix_len`` 2,064 leaves the last prefix
    block half full, so the first private write lands in a shared block."""
    suffix = np.random.default_rng(SEED_LENGTHS).integers(0, max_suffix + 1, size=num_seqs).astype(np.int32)
    rng = np.random.default_rng(SEED_VALUES)
    kv = (prefix_len, num_kv_heads, head_dim)
    pk = _normal(rng, kv, True)
    pv = _normal(rng, kv, True)
    sk, sv = [], []
    for s in suffix:
        sk.append(_normal(rng, (int(s) + 1, num_kv_heads, head_dim), True))
        sv.append(_normal(rng, (int(s) + 1, num_kv_heads, head_dim), True))
    q = _normal(rng, (num_seqs, num_heads, head_dim), True)
    return SharedPrefixCase(prefix_len, suffix, block_size, num_blocks, num_heads, num_kv_heads,
                            head_dim, pk, pv, sk, sv, q, 1.0 / math.sqrt(head_dim))
