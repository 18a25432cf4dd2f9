"""Test-only physical-block allocator with ref counts and copy-on-write (oracle side).

Test infrastructure only (see ``oracle/__init__``).  Host policy is outside the
GPU path; this exists to produce and check block tables, slot mappings and the
copy pairs that the block-copy operation consumes.

Behaviour follows "vLLM 原理" §3.3-§3.4 (a pool of blocks with a free queue, a
used set and per-block ref counts; a decode step needs a new block exactly
when the sequence's new length leaves remainder 1 modulo the block size) and
the copy-on-write rule of §2.1 (a write into a block whose ref count exceeds 1
first moves the writer onto a fresh copy and drops the old block's count by
one).  Prefix hashing is not modelled.
"""

from __future__ import annotations

from collections import deque


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.block_size = block_size
        self.ref = [0] * num_blocks
        order = list(range(num_blocks)) if free_order is None else list(free_order)
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self.free = deque(order)
        self.used = set()

    # -- raw block moves -------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise MemoryError("no free block")
        b = self.free.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        self.used.add(b)
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.used.discard(b)
            self.free.append(b)

    # -- sequence-level operations ---------------------------------------
    def blocks_needed(self, num_tokens: int) -> int:
        return -(-num_tokens // self.block_size)

    def can_allocate(self, num_tokens: int) -> bool:
        return len(self.free) >= self.blocks_needed(num_tokens)

    def allocate(self, num_tokens: int) -> list:
        """Fresh table covering ``num_tokens`` positions."""
        if not self.can_allocate(num_tokens):
            raise MemoryError("not enough free blocks")
        return [self._take() for _ in range(self.blocks_needed(num_tokens))]

    def fork(self, table: list) -> list:
        """A second sequence sharing every block of ``table`` (parallel sampling)."""
        for b in table:
            self.ref[b] += 1
        return list(table)

    def needs_new_block(self, new_len: int) -> bool:
        """True iff the token that brought the sequence to ``new_len`` opens a block."""
        return new_len % self.block_size == 1 or self.block_size == 1

    def can_append(self, new_len: int) -> bool:
        return len(self.free) >= (1 if self.needs_new_block(new_len) else 0)

    def write_slot(self, table: list, pos: int):
        """Make position ``pos`` writable for the sequence owning ``table``.

        Grows the table when ``pos`` opens a new logical block; when the block
        holding ``pos`` is shared (ref count > 1) it copies it first.  Returns
        ``(slot, copy_pair_or_None)`` with ``slot = block * block_size +
        offset``; ``table`` is updated in place.
        """
        lb, off = divmod(pos, self.block_size)
        if lb > len(table):
            raise ValueError("positions must be written in order")
        if lb == len(table):
            table.append(self._take())
        pair = None
        b = table[lb]
        if self.ref[b] > 1:
            nb = self._take()
            pair = (b, nb)
            self.ref[b] -= 1
            table[lb] = nb
            b = nb
        return b * self.block_size + off, pair

    def deallocate(self, table: list) -> None:
        for b in reversed(table):
            self._release(b)
        table.clear()
