"""Planted mistakes in the page-table simulator must fail at least one pin.

Each mutant is a plausible error in ``oracle.paged_pool`` (wrong reuse order,
a missing or needless copy-on-write, fills taken over the wrong sharer, a
preflight that forgets the private copy); it is planted on the CPU for one
test, and every pin of ``tests/test_oracle_pool.py`` is run against it.
"""

import pytest

import oracle.paged_pool as P
import test_oracle_pool as pins


def _release_to_bottom(self, seq):
    _, pages = self._lookup(seq)
    del self._length[seq], self._pages[seq]
    for b in pages:
        self._refcount[b] -= 1
        if self._refcount[b] == 0:
            self._stack.insert(0, b)            # FIFO reuse


def _never_copy(self, length, pages):
    return False


def _copy_full_blocks_too(self, length, pages):
    return bool(pages) and self._refcount[pages[-1]] > 1


def _fill_min_over_sharers(self):
    B = self.block_size
    fill = {}
    for seq, pages in self._pages.items():
        n = self._length[seq]
        for j, b in enumerate(pages):
            c = min(B, n - j * B)
            fill[b] = min(fill.get(b, c), c)
    return fill


_orig_append = P.PagedKVPool.append


def _preflight_ignores_copy(self, seq, token_count):
    length, pages = self._lookup(seq)
    grow = P.blocks_for(length + token_count, self.block_size) - len(pages)
    if grow > len(self._stack):
        raise MemoryError("short")
    if grow + 1 > len(self._stack) and token_count > 0 and self._tail_needs_copy(length, pages):
        # copies into a block it does not have: take the shared block's place without a replacement
        self._length[seq] = length + token_count
        pages.extend(self._take_ids(grow))
        return
    _orig_append(self, seq, token_count)


def _share_one_block_short(self, source, target, prefix_tokens):
    src_len, src_pages = self._lookup(source)
    if prefix_tokens > src_len:
        raise ValueError("too long")
    pages = src_pages[:prefix_tokens // self.block_size]      # floor instead of ceil
    for b in pages:
        self._refcount[b] += 1
    self._length[target] = prefix_tokens
    self._pages[target] = list(pages)


MUTANTS = {
    "fifo_reuse": ("release", _release_to_bottom),
    "no_copy_on_write": ("_tail_needs_copy", _never_copy),
    "copy_on_write_of_full_block": ("_tail_needs_copy", _copy_full_blocks_too),
    "fill_min_over_sharers": ("_fills", _fill_min_over_sharers),
    "preflight_ignores_copy": ("append", _preflight_ignores_copy),
    "share_prefix_floor": ("share_prefix", _share_one_block_short),
}

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and callable(getattr(pins, n))]


def _run(pin):
    if pin.__name__ == "test_short_child_survives_parent":
        for action, payload in (("release", 1), ("append", 5)):
            pin(action, payload)
    else:
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pool_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(P.PagedKVPool, attr, fn)
    failed = []
    for pin in PINS:
        try:
            _run(pin)
        except (AssertionError, ValueError, KeyError, MemoryError, IndexError, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"


def test_pins_pass_unmutated():
    for pin in PINS:
        _run(pin)
