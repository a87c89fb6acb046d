"""Pins of the page-table simulator against what the notebook fixes.

Sources: "Notebook 10. KV cache and serving: bytes, pages, and ceilings",
section 6 (the 8-block trace at block size 4, with the snapshot values of the
embedded contract in ``tests/golden/notebook10_contract.json``), section 9
(negative tests: OOM leaves the pool unchanged, a short child survives its
parent's release or copy-on-write, 2048 tokens at block size 16 waste
nothing) and the lecture-level core (private pages).
"""

import json
import os
import random

import pytest

from oracle.paged_pool import PagedKVPool, PrivatePagedKV

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "notebook10_contract.json")))


def run_trace(pool):
    """The section 6 trace; returns the snapshots after each step."""
    snaps = {}
    pool.create("A")
    pool.append("A", 6)
    snaps["after_a"] = pool.snapshot()
    pool.share_prefix("A", "B", 6)
    snaps["after_share"] = pool.snapshot()
    pool.append("B", 3)
    snaps["after_b_append"] = pool.snapshot()
    snaps["tables_after_b"] = (pool.page_table("A"), pool.page_table("B"))
    snaps["pairs_after_b"] = pool.take_copy_pairs()
    pool.release("A")
    snaps["after_a_release"] = pool.snapshot()
    return snaps


def test_trace_matches_notebook_contract():
    pool = PagedKVPool(GOLDEN["paged_trace_total_blocks"], GOLDEN["paged_trace_block_size"])
    snaps = run_trace(pool)
    for key in ("after_a", "after_share", "after_b_append", "after_a_release"):
        assert snaps[key] == GOLDEN["paged_trace"][key], key
    a, b = snaps["tables_after_b"]
    # The writer got a private copy of the shared partial block.
    assert a[-1] != b[1]


def test_trace_records_the_copy_on_write_pair():
    pool = PagedKVPool(8, 4)
    snaps = run_trace(pool)
    # A's partial block 1 was shared; B's private replacement is block 2.
    assert snaps["pairs_after_b"] == [(1, 2)]


def test_trace_is_relabelled_by_pop_order():
    """Handing out ids in another order only renames blocks (invariance)."""
    perm = [5, 2, 7, 0, 3, 6, 1, 4]
    pool = PagedKVPool(8, 4, pop_order=perm)
    snaps = run_trace(pool)
    for key in ("after_a", "after_share", "after_b_append", "after_a_release"):
        want = json.loads(json.dumps(GOLDEN["paged_trace"][key]))
        for s in want["sequences"].values():
            s["blocks"] = [perm[b] for b in s["blocks"]]
        assert snaps[key] == want, key
    assert snaps["pairs_after_b"] == [(perm[1], perm[2])]


def test_negative_cases_of_section_9():
    pool = PagedKVPool(2, 4)
    with pytest.raises(KeyError):
        pool.append("missing", 1)
    pool.create("x")
    with pytest.raises(ValueError):
        pool.create("x")
    pool.append("x", 6)
    before = pool.snapshot()
    with pytest.raises(MemoryError):
        pool.append("x", 3)
    assert pool.snapshot() == before
    with pytest.raises(ValueError):
        pool.share_prefix("x", "y", 7)
    with pytest.raises(ValueError):
        pool.append("x", -1)
    with pytest.raises(ValueError):
        pool.append("x", True)
    pool.validate()


def test_oom_preflight_counts_the_copy_on_write_block():
    """Appending into a shared partial block needs the replacement block too."""
    pool = PagedKVPool(2, 4)
    pool.create("p")
    pool.append("p", 2)                 # block 0, partial
    pool.share_prefix("p", "c", 2)      # shared partial block
    pool.create("q")
    pool.append("q", 4)                 # takes the last free block
    before = pool.snapshot()
    with pytest.raises(MemoryError):
        pool.append("c", 1)             # needs a private copy, none free
    assert pool.snapshot() == before
    assert pool.copy_pairs == []


@pytest.mark.parametrize("action,payload", [("release", 1), ("append", 5)])
def test_short_child_survives_parent(action, payload):
    pool = PagedKVPool(4, 4)
    pool.create("parent")
    pool.append("parent", 3)
    pool.share_prefix("parent", "child", 1)
    if action == "release":
        pool.release("parent")
    else:
        pool.append("parent", 1)
    assert pool.physical_payload_tokens == payload
    pool.append("child", 2)
    pool.validate()


def test_exact_2048_tokens_waste_nothing():
    pool = PagedKVPool(128, 16)
    pool.create("fixed")
    pool.append("fixed", 2048)
    assert pool.internal_waste_tokens == GOLDEN["exact_2048_waste_fraction"] * 2048 == 0
    assert pool.free_blocks == 0


def test_lecture_private_pages():
    pages = PrivatePagedKV(128, 16)
    pages.append_to("a", 2048)
    assert len(pages.tables["a"]) == 128
    before = (list(pages.free), dict(pages.lengths), {k: list(v) for k, v in pages.tables.items()})
    with pytest.raises(MemoryError):
        pages.append_to("a", 2049)
    assert before == (pages.free, pages.lengths, pages.tables)
    pages.release("a")
    assert len(pages.free) == 128
    with pytest.raises(ValueError):
        pages.append_to("x", -1)


def test_slots_follow_the_block_table():
    pool = PagedKVPool(16, 16, pop_order=list(range(15, -1, -1)))
    pool.create("s")
    pool.append("s", 40)
    table = pool.page_table("s")
    assert table == (15, 14, 13)
    assert pool.slots("s", 0, 3) == [15 * 16, 15 * 16 + 1, 15 * 16 + 2]
    assert pool.slots("s", 16, 1) == [14 * 16]
    assert pool.slots("s", 39, 1) == [13 * 16 + 7]


def test_random_operations_keep_invariants_and_fill_accounting():
    """Fuzz: every state reached obeys validate(); payload equals the number
    of distinct (block, slot) pairs any sequence covers (brute force)."""
    rng = random.Random(7)
    for trial in range(30):
        B = rng.choice([1, 2, 4, 16])
        pool = PagedKVPool(rng.randint(4, 24), B)
        names = []
        for step in range(40):
            op = rng.random()
            try:
                if op < 0.25 or not names:
                    n = f"s{trial}_{step}"
                    pool.create(n)
                    names.append(n)
                elif op < 0.6:
                    pool.append(rng.choice(names), rng.randint(0, 2 * B + 1))
                elif op < 0.8:
                    src = rng.choice(names)
                    t = f"c{trial}_{step}"
                    pool.share_prefix(src, t, rng.randint(0, pool.sequence_length(src)))
                    names.append(t)
                else:
                    n = rng.choice(names)
                    pool.release(n)
                    names.remove(n)
            except MemoryError:
                pass
            pool.validate()
            covered = set()
            for n in names:
                length = pool.sequence_length(n)
                for t in range(length):
                    covered.add(pool.slots(n, t, 1)[0])
            assert pool.physical_payload_tokens == len(covered)
            assert pool.logical_tokens == sum(pool.sequence_length(n) for n in names)


def test_released_blocks_are_handed_out_last_in_first_out():
    """Section 5: released blocks go back on top of the free stack, so the
    block freed last is the next one handed out."""
    pool = PagedKVPool(6, 4)
    for s, n in (("a", 4), ("b", 8), ("c", 4)):   # a: [0], b: [1, 2], c: [3]
        pool.create(s)
        pool.append(s, n)
    pool.release("b")                            # pushes 1, then 2
    pool.create("d")
    pool.append("d", 12)
    assert pool.page_table("d") == (2, 1, 4)
    pool.release("a")
    pool.release("c")
    pool.create("e")
    pool.append("e", 5)
    assert pool.page_table("e") == (3, 0)


def test_full_shared_block_is_never_copied():
    """Section 5: copy-on-write applies only to a shared *partial* last block;
    appending after a shared full block starts a new block and copies nothing
    (the 4096-token shared prefix is 256 full blocks: zero copy pairs)."""
    pool = PagedKVPool(8, 4)
    pool.create("root")
    pool.append("root", 8)
    pool.share_prefix("root", "x", 8)
    pool.append("x", 1)
    assert pool.take_copy_pairs() == []
    assert pool.page_table("x") == (0, 1, 2)
    pool.share_prefix("x", "y", 9)               # shares x's partial last block 2
    pool.append("y", 1)
    assert pool.take_copy_pairs() == [(2, 3)]
    assert pool.page_table("y") == (0, 1, 3) and pool.page_table("x") == (0, 1, 2)
    pool.validate()
