"""Page-table simulator: reference-counted physical blocks, prefix sharing and
copy-on-write. Test infrastructure: only the tests, the smoke check and the
benchmark's CPU legs use it.

Behaviour follows "Notebook 10. KV cache and serving: bytes, pages, and
ceilings": the page pool of section 5 (prefix sharing and copy-on-write), the
eight-block trace of section 6 and the negative tests of section 9. The pool
holds no tensor data. Logical token ``t`` of a sequence lives in physical
block ``table[t // B]`` at slot ``t % B``.

How this simulator is organised (its own design, not the notebook's code):

* State is only what cannot be derived: each sequence's length and page
  table, each block's reference count, and the free-id stack. How full a
  block is, the payload, the waste and the sharing savings are derived from
  the tables whenever they are asked for.
* Every mutation is first turned into a plan (the number of ids it takes
  from the stack and whether the last block must be privatised), the plan
  is checked, and only then applied. A refused plan changes nothing, which is
  the section 5 guarantee that running out of blocks never leaves a
  half-applied append.

Rules the pages fix, and the pins check:

* The free ids are a last-in first-out stack. A fresh pool hands out
  ``0, 1, 2, ...`` in that order; a released block goes on top and is the
  next one handed out.
* Appending to a sequence whose last block is partly filled *and* held by
  another sequence first gives the writer a private replacement holding the
  same filled slots (copy-on-write). A full shared block is never copied:
  new tokens start a new block.
* ``share_prefix`` hands the target the source's first ``ceil(prefix / B)``
  blocks, one more reference each.
* A block's fill is the largest number of its slots that any of its
  sharers covers (sharers may have different lengths).

Addition for a real cache: each copy-on-write records ``(old, new)`` in
``copy_pairs``; the block-copy kernel must move those blocks before the step's
append writes into ``new``.
"""

from __future__ import annotations

from typing import Hashable, Iterable


def _count(name: str, value, minimum: int) -> int:
    """A plain ``int`` no smaller than ``minimum`` (bools are refused)."""
    if isinstance(value, bool) or not isinstance(value, int) or value < minimum:
        raise ValueError(f"{name}: expected an int >= {minimum}, got {value!r}")
    return value


def blocks_for(tokens: int, block_size: int) -> int:
    """Blocks that hold ``tokens`` tokens: ceil(tokens / B) (0 for none)."""
    return -(-tokens // block_size)


class PagedKVPool:
    """Reference-counted block pool with prefix sharing and copy-on-write.

    ``pop_order`` (optional) is the order in which a fresh pool hands out
    block ids; by default ``0, 1, 2, ...`` as in the notebook. Another
    permutation only renames the physical ids (the invariance the attention
    kernels must respect).
    """

    def __init__(self, total_blocks: int, block_size: int = 16,
                 pop_order: Iterable[int] | None = None) -> None:
        self.total_blocks = _count("total_blocks", total_blocks, 1)
        self.block_size = _count("block_size", block_size, 1)
        hand_out = list(range(total_blocks)) if pop_order is None else [int(b) for b in pop_order]
        if sorted(hand_out) != list(range(total_blocks)):
            raise ValueError("pop_order: expected a permutation of 0 .. total_blocks - 1")
        # top of the stack (the next id handed out) is the end of the list
        self._stack: list[int] = hand_out[::-1]
        self._refcount = [0] * total_blocks
        self._length: dict[Hashable, int] = {}
        self._pages: dict[Hashable, list[int]] = {}
        self.copy_pairs: list[tuple[int, int]] = []

    # ------------------------------------------------------------ internals
    def _lookup(self, seq: Hashable) -> tuple[int, list[int]]:
        try:
            return self._length[seq], self._pages[seq]
        except KeyError:
            raise KeyError(f"no sequence {seq!r} in this pool") from None

    def _tail_needs_copy(self, length: int, pages: list[int]) -> bool:
        """Whether writing past ``length`` must first privatise the last block."""
        return length % self.block_size != 0 and self._refcount[pages[-1]] > 1

    def _take_ids(self, n: int) -> list[int]:
        """Pop ``n`` ids off the stack (the caller has checked there are enough)."""
        taken = [self._stack.pop() for _ in range(n)]
        for b in taken:
            self._refcount[b] += 1
        return taken

    def _fills(self) -> dict[int, int]:
        """Derived fill of every referenced block: max over its sharers."""
        B = self.block_size
        fill: dict[int, int] = {}
        for seq, pages in self._pages.items():
            n = self._length[seq]
            for j, b in enumerate(pages):
                fill[b] = max(fill.get(b, 0), min(B, n - j * B))
        return fill

    # ------------------------------------------------------------ mutators
    def create(self, seq: Hashable) -> None:
        """Register an empty sequence (hashable, not yet registered)."""
        hash(seq)
        if seq in self._length:
            raise ValueError(f"sequence {seq!r} is already registered")
        self._length[seq] = 0
        self._pages[seq] = []

    def append(self, seq: Hashable, token_count: int) -> None:
        """Grow ``seq`` by ``token_count`` tokens.

        Raises ``MemoryError``, with nothing changed, when the stack holds
        fewer ids than the plan needs (a private copy of a shared partial
        last block, plus the blocks the new length adds).
        """
        count = _count("token_count", token_count, 0)
        length, pages = self._lookup(seq)
        # plan
        privatise = count > 0 and self._tail_needs_copy(length, pages)
        grow = blocks_for(length + count, self.block_size) - len(pages)
        cost = grow + int(privatise)
        if cost > len(self._stack):
            raise MemoryError(f"appending {count} tokens to {seq!r} takes {cost} blocks; "
                              f"only {len(self._stack)} are free")
        # apply
        if privatise:
            shared = pages[-1]
            self._refcount[shared] -= 1
            (pages[-1],) = self._take_ids(1)
            self.copy_pairs.append((shared, pages[-1]))
        pages.extend(self._take_ids(grow))
        self._length[seq] = length + count

    def share_prefix(self, source: Hashable, target: Hashable, prefix_tokens: int) -> None:
        """Register ``target`` holding the first ``prefix_tokens`` tokens of ``source``."""
        src_len, src_pages = self._lookup(source)
        prefix = _count("prefix_tokens", prefix_tokens, 0)
        if prefix > src_len:
            raise ValueError(f"{source!r} holds {src_len} tokens; cannot share {prefix}")
        hash(target)
        if target in self._length:
            raise ValueError(f"sequence {target!r} is already registered")
        pages = src_pages[:blocks_for(prefix, self.block_size)]
        for b in pages:
            self._refcount[b] += 1
        self._length[target] = prefix
        self._pages[target] = list(pages)

    def release(self, seq: Hashable) -> None:
        """Forget ``seq``; every block it held last goes back on the stack, in
        table order (so its last such block is handed out next)."""
        _, pages = self._lookup(seq)
        del self._length[seq], self._pages[seq]
        for b in pages:
            self._refcount[b] -= 1
            if self._refcount[b] == 0:
                self._stack.append(b)

    def take_copy_pairs(self) -> list[tuple[int, int]]:
        """The copy-on-write pairs recorded since the last call (then cleared)."""
        pairs, self.copy_pairs = self.copy_pairs, []
        return pairs

    # ------------------------------------------------------------ queries
    def sequence_length(self, seq: Hashable) -> int:
        return self._lookup(seq)[0]

    def page_table(self, seq: Hashable) -> tuple[int, ...]:
        return tuple(self._lookup(seq)[1])

    def slots(self, seq: Hashable, start: int, count: int) -> list[int]:
        """Slot ids ``block * B + offset`` of logical tokens ``start .. start+count-1``."""
        length, pages = self._lookup(seq)
        if start < 0 or count < 0 or start + count > length:
            raise ValueError(f"tokens {start} .. {start + count - 1} are not all inside {seq!r}")
        B = self.block_size
        return [pages[t // B] * B + t % B for t in range(start, start + count)]

    @property
    def free_blocks(self) -> int:
        return len(self._stack)

    @property
    def allocated_blocks(self) -> int:
        return self.total_blocks - len(self._stack)

    @property
    def physical_capacity_tokens(self) -> int:
        return self.allocated_blocks * self.block_size

    @property
    def physical_payload_tokens(self) -> int:
        return sum(self._fills().values())

    @property
    def logical_tokens(self) -> int:
        return sum(self._length.values())

    @property
    def internal_waste_tokens(self) -> int:
        return self.physical_capacity_tokens - self.physical_payload_tokens

    @property
    def sharing_savings_tokens(self) -> int:
        return self.logical_tokens - self.physical_payload_tokens

    def snapshot(self) -> dict:
        """Summary with the field names of the notebook's recorded trace."""
        payload = self.physical_payload_tokens
        return {
            "sequences": {str(s): {"length": self._length[s], "blocks": list(self._pages[s])}
                          for s in sorted(self._length, key=repr)},
            "allocated_blocks": self.allocated_blocks,
            "free_blocks": self.free_blocks,
            "physical_capacity_tokens": self.physical_capacity_tokens,
            "physical_payload_tokens": payload,
            "logical_tokens": self.logical_tokens,
            "internal_waste_tokens": self.physical_capacity_tokens - payload,
            "sharing_savings_tokens": self.logical_tokens - payload,
        }

    def validate(self) -> None:
        """Check the pool's invariants; raises ``AssertionError`` on the first broken one."""
        N, B = self.total_blocks, self.block_size
        on_stack = [0] * N
        for b in self._stack:
            if not 0 <= b < N:
                raise AssertionError(f"free stack holds id {b}, outside the pool")
            on_stack[b] += 1
        held = [0] * N
        for seq, pages in self._pages.items():
            n = self._length[seq]
            if n < 0 or len(pages) != blocks_for(n, B):
                raise AssertionError(f"{seq!r}: {len(pages)} blocks for {n} tokens")
            if len(set(pages)) != len(pages):
                raise AssertionError(f"{seq!r} maps one block twice")
            for b in pages:
                if not 0 <= b < N:
                    raise AssertionError(f"{seq!r} maps id {b}, outside the pool")
                held[b] += 1
        for b in range(N):
            if held[b] != self._refcount[b]:
                raise AssertionError(f"block {b}: reference count {self._refcount[b]}, held by {held[b]}")
            if on_stack[b] != (held[b] == 0):
                raise AssertionError(f"block {b}: held by {held[b]} tables, {on_stack[b]} times on the stack")
        for b, f in self._fills().items():
            if not 1 <= f <= B:
                raise AssertionError(f"block {b}: fill {f} outside 1 .. {B}")
        if self.logical_tokens < self.physical_payload_tokens:
            raise AssertionError("more tokens stored than the sequences hold")


class PrivatePagedKV:
    """Private pages only (the notebook's lecture-level core): no sharing, no
    copy. ``append_to(seq, total)`` grows a sequence to ``total`` tokens with
    all the blocks it needs from the stack, or none of them."""

    def __init__(self, n_blocks: int, block_size: int = 16) -> None:
        self.n_blocks = _count("n_blocks", n_blocks, 1)
        self.block_size = _count("block_size", block_size, 1)
        self.free = list(range(n_blocks - 1, -1, -1))
        self.tables: dict[Hashable, list[int]] = {}
        self.lengths: dict[Hashable, int] = {}

    def append_to(self, seq: Hashable, total_tokens: int) -> None:
        total = _count("total_tokens", total_tokens, 0)
        hash(seq)
        if total < self.lengths.get(seq, 0):
            raise ValueError(f"{seq!r} already holds more than {total} tokens")
        pages = self.tables.get(seq, [])
        extra = blocks_for(total, self.block_size) - len(pages)
        if extra > len(self.free):
            raise MemoryError(f"{seq!r} needs {extra} more blocks; only {len(self.free)} are free")
        self.tables[seq] = pages + [self.free.pop() for _ in range(extra)]
        self.lengths[seq] = total

    def release(self, seq: Hashable) -> None:
        self.free.extend(self.tables.pop(seq))
        del self.lengths[seq]
