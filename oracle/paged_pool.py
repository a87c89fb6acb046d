"""Page-table simulator: ref-counted physical blocks, prefix sharing, copy-on-write.

Restates the behaviour of the page pool of "Notebook 10. KV cache and serving:
bytes, pages, and ceilings", section 5 ("Page pool: prefix sharing and
copy-on-write") and its section 6 trace, in code written for this oracle. The
pool stores no tensors: it tracks, per physical block, a reference count and a
fill (live slots), and per sequence a logical length and a page table (list of
physical block ids; logical token ``t`` lives in ``table[t // B]`` at slot
``t % B``).

Behaviour that the pages fix and that the pins check:

* Free blocks form a stack. A fresh pool hands out ids in ascending order
  (the stack starts as ``N-1 ... 0`` and pops from the end); released blocks
  are pushed on top, so the most recently freed block is reused first.
* ``append`` first counts the blocks it needs (one copy-on-write replacement
  if the last block is partial *and* shared, plus enough new blocks for the
  overflow) and raises ``MemoryError`` before touching anything if the free
  stack is too short ("Allocation is preflighted, so OOM cannot leave a
  partially mutated pool").
* Copy-on-write happens only for a shared partial final block: the old block
  loses one reference and a fresh block with the same number of filled slots
  replaces it in the writer's table. A full shared block is never copied,
  since appends start a new block.
* ``share_prefix`` gives the target the source's first ``ceil(prefix/B)``
  blocks and adds one reference to each.
* A block's fill is the largest number of its slots that any sharer still
  covers (sharers of unequal length, notebook section 5).

The single addition for a real cache: every copy-on-write records the pair
``(old_block, new_block)`` in ``copy_pairs``. The block-copy kernel must copy
those blocks before the append writes into ``new_block``.
"""

from __future__ import annotations

import math
from typing import Hashable, Iterable


def _count(name: str, value, minimum: int) -> int:
    """Integer check that refuses bools (notebook section 1 validators)."""
    if isinstance(value, bool) or not isinstance(value, int) or value < minimum:
        raise ValueError(f"{name} must be an integer >= {minimum}")
    return value


class PagedKVPool:
    """Ref-counted block pool with prefix sharing and copy-on-write.

    ``pop_order`` (optional) is the order in which a fresh pool hands out
    block ids; by default ``0, 1, 2, ...`` exactly as the notebook's pool.
    Passing a permutation relabels the physical ids without changing any
    other behaviour (the invariance the decode kernel must respect).
    """

    def __init__(self, total_blocks: int, block_size: int = 16,
                 pop_order: Iterable[int] | None = None) -> None:
        self.total_blocks = _count("total_blocks", total_blocks, 1)
        self.block_size = _count("block_size", block_size, 1)
        order = list(range(self.total_blocks)) if pop_order is None else [int(b) for b in pop_order]
        if sorted(order) != list(range(self.total_blocks)):
            raise ValueError("pop_order must be a permutation of the block ids")
        # The stack pops from its end, so store the hand-out order reversed.
        self._free: list[int] = order[::-1]
        self._refs = [0] * self.total_blocks
        self._fill = [0] * self.total_blocks
        self._len: dict[Hashable, int] = {}
        self._table: dict[Hashable, list[int]] = {}
        self.copy_pairs: list[tuple[int, int]] = []

    # ------------------------------------------------------------ helpers
    def _state(self, seq: Hashable) -> tuple[int, list[int]]:
        if seq not in self._len:
            raise KeyError(f"unknown sequence: {seq!r}")
        return self._len[seq], self._table[seq]

    def _pop_block(self, filled: int) -> int:
        block = self._free.pop()
        self._refs[block] = 1
        self._fill[block] = filled
        return block

    def _needed_blocks(self, length: int, table: list[int], count: int) -> int:
        """Blocks an append of ``count`` tokens must take from the free stack."""
        if count == 0:
            return 0
        B = self.block_size
        used_in_last = length % B
        room = 0
        need = 0
        if table and used_in_last:
            room = B - used_in_last
            if self._refs[table[-1]] > 1:
                need += 1  # private replacement for the shared partial block
        overflow = max(0, count - room)
        return need + (overflow + B - 1) // B

    def _recount_fills(self) -> None:
        """Fill of a block = max over its sharers of the slots they cover."""
        B = self.block_size
        fills = [0] * self.total_blocks
        for seq, table in self._table.items():
            n = self._len[seq]
            for j, block in enumerate(table):
                covered = min(B, n - j * B)
                if covered > fills[block]:
                    fills[block] = covered
        self._fill = fills

    # ------------------------------------------------------------ mutators
    def create(self, seq: Hashable) -> None:
        """Register an empty sequence; ids must be hashable and unique."""
        hash(seq)
        if seq in self._len:
            raise ValueError(f"sequence already exists: {seq!r}")
        self._len[seq] = 0
        self._table[seq] = []

    def append(self, seq: Hashable, token_count: int) -> None:
        """Grow ``seq`` by ``token_count`` logical tokens.

        Raises ``MemoryError`` with the pool unchanged when the free stack
        cannot cover the copy-on-write replacement plus the new blocks.
        """
        count = _count("token_count", token_count, 0)
        length, table = self._state(seq)
        need = self._needed_blocks(length, table, count)
        if need > len(self._free):
            raise MemoryError(f"need {need} free blocks, {len(self._free)} remain")
        if count == 0:
            return
        B = self.block_size
        used_in_last = length % B
        if table and used_in_last:
            last = table[-1]
            if self._refs[last] > 1:
                self._refs[last] -= 1
                fresh = self._pop_block(filled=used_in_last)
                table[-1] = fresh
                self.copy_pairs.append((last, fresh))
                last = fresh
            take = min(count, B - used_in_last)
            self._fill[last] = used_in_last + take
            length += take
            count -= take
        while count > 0:
            take = min(count, B)
            table.append(self._pop_block(filled=take))
            length += take
            count -= take
        self._len[seq] = length
        self._recount_fills()
        self.validate()

    def share_prefix(self, source: Hashable, target: Hashable, prefix_tokens: int) -> None:
        """Create ``target`` whose first ``prefix_tokens`` tokens are ``source``'s."""
        src_len, src_table = self._state(source)
        prefix = _count("prefix_tokens", prefix_tokens, 0)
        if prefix > src_len:
            raise ValueError("prefix_tokens exceeds source length")
        if target in self._len:
            raise ValueError(f"target sequence already exists: {target!r}")
        hash(target)
        shared = src_table[: -(-prefix // self.block_size)] if prefix else []
        for block in shared:
            self._refs[block] += 1
        self._len[target] = prefix
        self._table[target] = list(shared)
        self.validate()

    def release(self, seq: Hashable) -> None:
        """Drop ``seq``; blocks whose last reference goes are cleared and pushed."""
        _, table = self._state(seq)
        for block in table:
            self._refs[block] -= 1
            if self._refs[block] == 0:
                self._fill[block] = 0
                self._free.append(block)
        del self._len[seq]
        del self._table[seq]
        self._recount_fills()
        self.validate()

    def take_copy_pairs(self) -> list[tuple[int, int]]:
        """Return and clear the copy-on-write pairs recorded so far."""
        pairs, self.copy_pairs = self.copy_pairs, []
        return pairs

    # ------------------------------------------------------------ queries
    def sequence_length(self, seq: Hashable) -> int:
        return self._state(seq)[0]

    def page_table(self, seq: Hashable) -> tuple[int, ...]:
        return tuple(self._state(seq)[1])

    def slots(self, seq: Hashable, start: int, count: int) -> list[int]:
        """Physical slot ids ``block * B + offset`` of logical tokens [start, start+count)."""
        length, table = self._state(seq)
        if start < 0 or start + count > length:
            raise ValueError("token range outside the sequence")
        B = self.block_size
        return [table[t // B] * B + t % B for t in range(start, start + count)]

    @property
    def free_blocks(self) -> int:
        return len(self._free)

    @property
    def allocated_blocks(self) -> int:
        return self.total_blocks - len(self._free)

    @property
    def physical_capacity_tokens(self) -> int:
        return self.allocated_blocks * self.block_size

    @property
    def physical_payload_tokens(self) -> int:
        return sum(f for f, r in zip(self._fill, self._refs) if r)

    @property
    def logical_tokens(self) -> int:
        return sum(self._len.values())

    @property
    def internal_waste_tokens(self) -> int:
        return self.physical_capacity_tokens - self.physical_payload_tokens

    @property
    def sharing_savings_tokens(self) -> int:
        return self.logical_tokens - self.physical_payload_tokens

    def snapshot(self) -> dict:
        """Deterministic summary with the notebook's field names."""
        seqs = sorted(self._len, key=repr)
        return {
            "sequences": {str(s): {"length": self._len[s], "blocks": list(self._table[s])}
                          for s in seqs},
            "allocated_blocks": self.allocated_blocks,
            "free_blocks": self.free_blocks,
            "physical_capacity_tokens": self.physical_capacity_tokens,
            "physical_payload_tokens": self.physical_payload_tokens,
            "logical_tokens": self.logical_tokens,
            "internal_waste_tokens": self.internal_waste_tokens,
            "sharing_savings_tokens": self.sharing_savings_tokens,
        }

    def validate(self) -> None:
        """Invariants of notebook section 5: tables, references, fills, free stack."""
        if len(set(self._free)) != len(self._free):
            raise AssertionError("free stack holds a block twice")
        if any(not 0 <= b < self.total_blocks for b in self._free):
            raise AssertionError("free stack holds an invalid id")
        refs = [0] * self.total_blocks
        for seq, table in self._table.items():
            n = self._len[seq]
            if n < 0:
                raise AssertionError("negative sequence length")
            if len(table) != -(-n // self.block_size):
                raise AssertionError("page table length disagrees with sequence length")
            if len(set(table)) != len(table):
                raise AssertionError("a sequence maps one block twice")
            for b in table:
                if not 0 <= b < self.total_blocks:
                    raise AssertionError("page table holds an invalid id")
                refs[b] += 1
        free = set(self._free)
        for b in range(self.total_blocks):
            if refs[b] != self._refs[b]:
                raise AssertionError("reference count disagrees with page tables")
            if refs[b] == 0:
                if b not in free or self._fill[b] != 0:
                    raise AssertionError("unreferenced block is not clean and free")
            else:
                if b in free:
                    raise AssertionError("referenced block sits on the free stack")
                if not 1 <= self._fill[b] <= self.block_size:
                    raise AssertionError("referenced block has an invalid fill")
        if self.logical_tokens < self.physical_payload_tokens:
            raise AssertionError("physical payload exceeds logical payload")


class PrivatePagedKV:
    """Private pages only (notebook "Lecture-level core"): no sharing, no copy.

    ``append_to(seq, total)`` grows a sequence to ``total`` tokens, taking
    ``ceil(total/B) - len(table)`` blocks from the free stack, all or none.
    """

    def __init__(self, n_blocks: int, block_size: int = 16) -> None:
        self.n_blocks = _count("n_blocks", n_blocks, 1)
        self.block_size = _count("block_size", block_size, 1)
        self.free = list(range(self.n_blocks))[::-1]
        self.tables: dict[Hashable, list[int]] = {}
        self.lengths: dict[Hashable, int] = {}

    def append_to(self, seq: Hashable, total_tokens: int) -> None:
        total = _count("total_tokens", total_tokens, 0)
        hash(seq)
        if total < self.lengths.get(seq, 0):
            raise ValueError("append_to cannot shorten a sequence")
        table = self.tables.get(seq, [])
        need = -(-total // self.block_size) - len(table)
        if need > len(self.free):
            raise MemoryError("not enough free blocks")
        self.tables[seq] = table
        for _ in range(need):
            table.append(self.free.pop())
        self.lengths[seq] = total

    def release(self, seq: Hashable) -> None:
        self.free.extend(self.tables.pop(seq))
        del self.lengths[seq]


def blocks_for(tokens: int, block_size: int) -> int:
    """Number of blocks that hold ``tokens`` tokens: ceil(tokens / B)."""
    return math.ceil(tokens / block_size) if tokens else 0
