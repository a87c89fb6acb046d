"""The library's block pool (pkv_pool_*, host C++) against the notebook and
the oracle's page-pool simulator.

Sources: "Notebook 10. KV cache and serving: bytes, pages, and ceilings",
section 6 trace (golden fixture), section 9 negative cases, and a
differential fuzz against ``oracle.paged_pool.PagedKVPool``: after every
operation the two must agree on tables, lengths, slot ids, copy-on-write
pairs and every counter of the snapshot.
"""

import json
import os
import random

import numpy as np
import pytest

from oracle.paged_pool import PagedKVPool

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "notebook10_contract.json")))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_209_gb300 import build, pkv as P
    if not os.path.exists(P.LIB_PATH):
        build.build()
    P.load_library()
    return P


def snapshot(pool, names):
    st = pool.stats()
    snap = {k: st[k] for k in ("allocated_blocks", "free_blocks", "physical_capacity_tokens",
                               "physical_payload_tokens", "logical_tokens", "internal_waste_tokens",
                               "sharing_savings_tokens")}
    snap["sequences"] = {names[s]: {"length": pool.sequence_length(s), "blocks": list(pool.page_table(s))}
                         for s in sorted(names)}
    return snap


def test_trace_matches_notebook(pkv):
    A, B = 1, 2
    names = {A: "A"}
    pool = pkv.BlockPool(GOLDEN["paged_trace_total_blocks"], GOLDEN["paged_trace_block_size"])
    pool.add_sequence(A)
    slots, pair = pool.append(A, 6)
    assert list(slots) == [0, 1, 2, 3, 4, 5] and pair is None
    assert snapshot(pool, names) == GOLDEN["paged_trace"]["after_a"]
    pool.share_prefix(A, B, 6)
    names[B] = "B"
    assert snapshot(pool, names) == GOLDEN["paged_trace"]["after_share"]
    slots, pair = pool.append(B, 3)
    assert pair == (1, 2)                      # the shared partial block is copied
    assert list(slots) == [2 * 4 + 2, 2 * 4 + 3, 3 * 4 + 0]
    assert snapshot(pool, names) == GOLDEN["paged_trace"]["after_b_append"]
    assert pool.page_table(A)[-1] != pool.page_table(B)[1]
    pool.release(A)
    del names[A]
    assert snapshot(pool, names) == GOLDEN["paged_trace"]["after_a_release"]
    pool.validate()


def test_negative_cases(pkv):
    pool = pkv.BlockPool(2, 4)
    with pytest.raises(pkv.PkvError) as e:
        pool.append(7, 1)
    assert e.value.name == "PKV_ERR_UNKNOWN_SEQUENCE"
    pool.add_sequence(7)
    with pytest.raises(pkv.PkvError) as e:
        pool.add_sequence(7)
    assert e.value.name == "PKV_ERR_EXISTS"
    pool.append(7, 6)
    before = (pool.stats(), pool.page_table(7), pool.sequence_length(7))
    with pytest.raises(pkv.PkvError) as e:
        pool.append(7, 3)
    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
    assert (pool.stats(), pool.page_table(7), pool.sequence_length(7)) == before
    with pytest.raises(pkv.PkvError) as e:
        pool.share_prefix(7, 8, 7)
    assert e.value.name == "PKV_ERR_SHAPE"
    with pytest.raises(pkv.PkvError) as e:
        pool.append(7, -1)
    assert e.value.name == "PKV_ERR_SHAPE"
    with pytest.raises(pkv.PkvError) as e:
        pkv.BlockPool(4, 4, pop_order=[0, 1, 1, 2])
    assert e.value.name == "PKV_ERR_RANGE"
    pool.validate()


@pytest.mark.parametrize("action,payload", [("release", 1), ("append", 5)])
def test_short_child_survives_parent(pkv, action, payload):
    pool = pkv.BlockPool(4, 4)
    pool.add_sequence(1)
    pool.append(1, 3)
    pool.share_prefix(1, 2, 1)
    if action == "release":
        pool.release(1)
    else:
        pool.append(1, 1)
    assert pool.stats()["physical_payload_tokens"] == payload
    pool.append(2, 2)
    pool.validate()


def test_exact_2048_wastes_nothing(pkv):
    pool = pkv.BlockPool(128, 16)
    pool.add_sequence(0)
    pool.append(0, 2048)
    assert pool.stats()["internal_waste_tokens"] == 0 and pool.stats()["free_blocks"] == 0


def oracle_state(o, seqs):
    snap = o.snapshot()
    return {k: v for k, v in snap.items() if k != "sequences"}, {
        s: (o.sequence_length(s), tuple(o.page_table(s))) for s in seqs}


def pool_state(p, seqs):
    st = p.stats()
    keys = ("allocated_blocks", "free_blocks", "physical_capacity_tokens", "physical_payload_tokens",
            "logical_tokens", "internal_waste_tokens", "sharing_savings_tokens")
    return {k: st[k] for k in keys}, {s: (p.sequence_length(s), p.page_table(s)) for s in seqs}


@pytest.mark.parametrize("seed", range(12))
def test_differential_fuzz_against_the_oracle(pkv, seed):
    rng = random.Random(seed)
    B = rng.choice([1, 4, 16])
    N = rng.randint(6, 40)
    order = list(range(N))
    rng.shuffle(order)
    lib = pkv.BlockPool(N, B, pop_order=order)
    ora = PagedKVPool(N, B, pop_order=order)
    live, next_id = [], 0
    for step in range(120):
        op = rng.random()
        try:
            if op < 0.2 or not live:
                lib.add_sequence(next_id)
                ora.create(next_id)
                live.append(next_id)
                next_id += 1
            elif op < 0.6:
                s = rng.choice(live)
                n = rng.randint(0, 2 * B + 2)
                start = ora.sequence_length(s)
                try:
                    ora.append(s, n)
                except MemoryError:
                    with pytest.raises(pkv.PkvError) as e:
                        lib.append(s, n)
                    assert e.value.name == "PKV_ERR_OUT_OF_BLOCKS"
                    continue
                slots, pair = lib.append(s, n)
                assert list(slots) == ora.slots(s, start, n)
                assert ([pair] if pair else []) == ora.take_copy_pairs()
            elif op < 0.75:
                seqs = rng.sample(live, rng.randint(1, len(live)))
                want_slots, done = [], 0
                for s in seqs:
                    start = ora.sequence_length(s)
                    try:
                        ora.append(s, 1)
                    except MemoryError:
                        break
                    want_slots += ora.slots(s, start, 1)
                    done += 1
                want_pairs = ora.take_copy_pairs()
                if done < len(seqs):
                    with pytest.raises(pkv.PkvError):
                        lib.append_batch(seqs, [1] * len(seqs))
                else:
                    slots, pairs = lib.append_batch(seqs, [1] * len(seqs))
                    assert list(slots) == want_slots
                    assert [tuple(p) for p in pairs] == want_pairs
            elif op < 0.88:
                src = rng.choice(live)
                k = rng.randint(0, ora.sequence_length(src))
                lib.share_prefix(src, next_id, k)
                ora.share_prefix(src, next_id, k)
                live.append(next_id)
                next_id += 1
            else:
                s = rng.choice(live)
                lib.release(s)
                ora.release(s)
                live.remove(s)
        finally:
            pass
        assert pool_state(lib, live) == oracle_state(ora, live), (seed, step)
        lib.validate()


def test_block_tables_export(pkv):
    pool = pkv.BlockPool(64, 16, pop_order=np.random.default_rng(3).permutation(64))
    for s, n in ((10, 40), (11, 1), (12, 0), (13, 300)):
        pool.add_sequence(s)
        pool.append(s, n)
    tables, lens = pool.block_tables([13, 10, 12, 11], width=19)
    assert list(lens) == [300, 40, 0, 1]
    assert tuple(tables[1][:3]) == pool.page_table(10) and all(tables[1][3:] == -1)
    assert all(tables[2] == -1)
    with pytest.raises(pkv.PkvError) as e:
        pool.block_tables([13], width=18)     # 300 tokens need 19 blocks
    assert e.value.name == "PKV_ERR_SHAPE"
