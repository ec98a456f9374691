"""Host block manager: a seeded generator of block tables.

This is the pool / free list / reference count / per-request block table of
"19.2 KV Cache 系统化管理" §19.2.3 (``PhysicalBlockPool``, ``BlockTable``)
together with fork and copy-on-write from §19.2.2 and from
"企业官网建设流程全解析" §4.2 / §5.1 (the child's table is a prefix copy of
the parent's and every shared block's count goes up).  It runs on the host
and only produces inputs for the device path: block tables, context lengths,
token positions and copy pairs.  It holds no KV data.

Differences from the page's pool, on purpose:

* The free list is shuffled once with a seed, then popped from the end
  (the page pops ``list(range(n))`` from the end).  Scattered physical
  placement is what the device path has to cope with.
* ``append_token`` only reserves; the device writes the data.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np


class PoolExhausted(RuntimeError):
    """No free physical block is left (the page raises on exhaustion too)."""


class BlockPool:
    def __init__(self, num_blocks: int, seed: Optional[int] = None):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.num_blocks = int(num_blocks)
        order = np.arange(self.num_blocks)
        if seed is not None:
            order = np.random.default_rng(seed).permutation(self.num_blocks)
        self.free_list: List[int] = [int(b) for b in order]
        self.ref_counts = [0] * self.num_blocks

    # -- allocation (LIFO pop, refcount 1) --------------------------------
    def allocate(self) -> int:
        if not self.free_list:
            raise PoolExhausted("physical block pool exhausted")
        b = self.free_list.pop()
        self.ref_counts[b] = 1
        return b

    def incref(self, b: int) -> None:
        if self.ref_counts[b] <= 0:
            raise RuntimeError(f"incref of free block {b}")
        self.ref_counts[b] += 1

    def release(self, b: int) -> None:
        if self.ref_counts[b] <= 0:
            raise RuntimeError(f"release of free block {b}")
        self.ref_counts[b] -= 1
        if self.ref_counts[b] == 0:
            self.free_list.append(b)

    @property
    def num_free(self) -> int:
        return len(self.free_list)

    @property
    def num_allocated(self) -> int:
        return sum(1 for c in self.ref_counts if c > 0)

    def check_invariants(self, tables: List["SeqBlocks"]) -> None:
        """Leak check and reference check ("企业官网建设流程全解析" §7.1,
        §7.2): allocated + free = pool size, no block is both, and each
        block's count is at least the number of tables that reference it."""
        free = set(self.free_list)
        if len(free) != len(self.free_list):
            raise AssertionError("duplicate entry in free list")
        alloc = {b for b, c in enumerate(self.ref_counts) if c > 0}
        if alloc & free:
            raise AssertionError("block both allocated and free")
        if len(alloc) + len(free) != self.num_blocks:
            raise AssertionError("leaked blocks: allocated + free != pool size")
        users = [0] * self.num_blocks
        for t in tables:
            for b in set(t.mapping):
                users[b] += 1
        for b in range(self.num_blocks):
            if self.ref_counts[b] < users[b]:
                raise AssertionError(f"block {b}: refcount {self.ref_counts[b]} < {users[b]} users")


@dataclass
class SeqBlocks:
    """Per-request block table: logical block i -> ``mapping[i]``."""

    pool: BlockPool
    block_size: int
    mapping: List[int] = field(default_factory=list)
    num_tokens: int = 0

    def grow_to(self, num_tokens: int) -> None:
        """Reserve blocks for ``num_tokens`` tokens (prefill of that many)."""
        while len(self.mapping) * self.block_size < num_tokens:
            self.mapping.append(self.pool.allocate())
        self.num_tokens = max(self.num_tokens, num_tokens)

    def share_prefix(self, other: "SeqBlocks", num_blocks: int) -> None:
        """Point the first ``num_blocks`` logical blocks at ``other``'s
        physical blocks (whole blocks only) and count the new references."""
        if self.mapping:
            raise RuntimeError("share_prefix on a non-empty table")
        for b in other.mapping[:num_blocks]:
            self.pool.incref(b)
            self.mapping.append(b)
        self.num_tokens = num_blocks * self.block_size

    def fork(self) -> "SeqBlocks":
        child = SeqBlocks(self.pool, self.block_size, list(self.mapping), self.num_tokens)
        for b in child.mapping:
            self.pool.incref(b)
        return child

    def append_token(self) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot for one more token.

        Returns ``(position, copy_pair)``.  A token that opens a new logical
        block gets a fresh block.  A token that goes into a partially filled
        block that other tables share triggers copy-on-write: a new block is
        allocated, ``(old, new)`` is returned for the device copy, this table
        is repointed and the old block's count drops by one.
        """
        pos = self.num_tokens
        pair = None
        if pos % self.block_size == 0 and pos // self.block_size == len(self.mapping):
            self.mapping.append(self.pool.allocate())
        else:
            last = self.mapping[pos // self.block_size]
            if self.pool.ref_counts[last] > 1:
                new = self.pool.allocate()
                pair = (last, new)
                self.mapping[pos // self.block_size] = new
                self.pool.release(last)
        self.num_tokens += 1
        return pos, pair

    def release_all(self) -> None:
        for b in self.mapping:
            self.pool.release(b)
        self.mapping.clear()
        self.num_tokens = 0


def _move_all(seq: SeqBlocks, to_pool: BlockPool) -> List[Tuple[int, int]]:
    need = len(seq.mapping)
    if to_pool.num_free < need:
        raise PoolExhausted(f"need {need} free blocks, {to_pool.num_free} left")
    pairs = [(b, to_pool.allocate()) for b in seq.mapping]
    for b in seq.mapping:
        seq.pool.release(b)
    seq.mapping = [d for _, d in pairs]
    seq.pool = to_pool
    return pairs


def swap_out(seq: SeqBlocks, host_pool: BlockPool) -> List[Tuple[int, int]]:
    """Preempt a request by swapping ("19.2 KV Cache 系统化管理" §19.2.6):
    every one of its blocks at once (all or nothing) gets a block of the
    host pool, its GPU blocks are released, and its table is repointed to the
    host blocks.  Returns the ``(gpu_block, host_block)`` pairs the device
    swap must copy before the released GPU blocks are reused.  A block shared
    with other tables keeps their references; this request leaves with its
    own copy.  Raises ``PoolExhausted`` (and changes nothing) when the host
    pool lacks room."""
    return _move_all(seq, host_pool)


def swap_in(seq: SeqBlocks, gpu_pool: BlockPool) -> List[Tuple[int, int]]:
    """Resume a swapped-out request: fresh GPU blocks for all of its host
    blocks (all or nothing), host blocks released.  Returns the
    ``(host_block, gpu_block)`` pairs to copy."""
    return _move_all(seq, gpu_pool)
