"""Inputs for the GPU parity tests, built on the CPU.

Index metadata (tables, lengths, slot mappings, copy pairs) for the
workloads with sharing comes from the oracle's page-pool simulator, so the
copy-on-write pairs are the ones the notebook's rules produce. Values are
seeded draws from ``paged_kv_cache_209_gb300.workloads``. Nothing here calls
the CUDA library.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle.paged_pool import PagedKVPool
from paged_kv_cache_209_gb300 import workloads as W

B = 16


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_view(t: torch.Tensor) -> np.ndarray:
    """Host numpy view the oracle reads: float32 values or bf16 bits."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().numpy()


def dtype_name(t: torch.Tensor) -> str:
    return "bf16" if t.dtype == torch.bfloat16 else "f32"


def padded_tables(pool: PagedKVPool, seqs, width: int | None = None) -> np.ndarray:
    tabs = [list(pool.page_table(s)) for s in seqs]
    w = width or max(1, max(len(t) for t in tabs))
    out = np.full((len(seqs), w), -1, dtype=np.int32)
    for i, t in enumerate(tabs):
        out[i, :len(t)] = t
    return out


def simulate_workload_step(tables, lens_after, queries, num_blocks, shared_blocks=0):
    """Rebuild a full-size workload's cache state with the oracle's page pool
    and run the step's appends there.

    Before the step sequence i holds ``lens_after[i] - queries`` tokens; the
    step appends ``queries`` tokens to each sequence in index order. With
    ``shared_blocks`` > 0 a root sequence holds that many full blocks and
    every sequence starts as a copy of it (``share_prefix``). The pool hands
    out ids in the order these operations request them, read off ``tables``,
    so the simulator must end with exactly ``tables`` (asserted: the
    workload's tables are a state the pool's rules can reach).

    Returns ``(slots int64 [batch * queries] in sequence order, copy pairs
    int64 [n][2])`` as the oracle's pool produces them.
    """
    tables = np.asarray(tables)
    lens_after = np.asarray(lens_after, dtype=np.int64)
    before = lens_after - queries
    nb_before, nb_after = W.blocks_needed(before), W.blocks_needed(lens_after)
    order = [int(b) for b in tables[0, :shared_blocks]] if shared_blocks else []
    for i in range(len(lens_after)):
        order += [int(b) for b in tables[i, shared_blocks:nb_before[i]]]
    for i in range(len(lens_after)):
        order += [int(b) for b in tables[i, nb_before[i]:nb_after[i]]]
    taken = set(order)
    assert len(taken) == len(order), "a block id is requested twice"
    order += [b for b in range(num_blocks) if b not in taken]
    pool = PagedKVPool(num_blocks, B, pop_order=order)
    if shared_blocks:
        pool.create("root")
        pool.append("root", shared_blocks * B)
    for i in range(len(lens_after)):
        if shared_blocks:
            pool.share_prefix("root", i, shared_blocks * B)
        else:
            pool.create(i)
        pool.append(i, int(before[i]) - shared_blocks * B)
    slots = []
    for i in range(len(lens_after)):
        start = pool.sequence_length(i)
        pool.append(i, queries)
        slots += pool.slots(i, start, queries)
    pairs = np.array(pool.take_copy_pairs(), dtype=np.int64).reshape(-1, 2)
    got = padded_tables(pool, range(len(lens_after)), width=tables.shape[1])
    assert np.array_equal(got, tables), "the page pool does not reach the workload's tables"
    return np.array(slots, dtype=np.int64), pairs


def tiny_case(dtype=torch.float32, head_dim=64, q_heads=4, kv_heads=2, poison=False):
    """The 3-sequence workload: seq 1 holds 9 tokens, seq 0 shares its first 6
    (a shared partial block), seq 2 holds 33; then one step appends one token
    to each sequence in index order (seq 0 copies the shared block first)."""
    cfg = W.CONFIGS["tiny_f32"]
    perm = np.random.default_rng(cfg["seed"]).permutation(cfg["num_blocks"])
    pool = PagedKVPool(cfg["num_blocks"], B, pop_order=perm)
    pool.create(1)
    pool.append(1, 9)
    pool.share_prefix(1, 0, 6)
    pool.create(2)
    pool.append(2, 33)
    seqs = [0, 1, 2]
    lens_before = np.array([pool.sequence_length(s) for s in seqs], dtype=np.int32)
    tables_before = padded_tables(pool, seqs, width=4)
    slots = []
    for s in seqs:
        n = pool.sequence_length(s)
        pool.append(s, 1)
        slots.append(pool.slots(s, n, 1)[0])
    pairs = pool.take_copy_pairs()
    lens_after = np.array([pool.sequence_length(s) for s in seqs], dtype=np.int32)
    tables_after = padded_tables(pool, seqs, width=4)
    nb = cfg["num_blocks"]
    kp = W.numpy_normal((nb, kv_heads, B, head_dim), 101)
    vp = W.numpy_normal((nb, kv_heads, B, head_dim), 102)
    if poison:
        used = set()
        for i, s in enumerate(seqs):
            for t in range(int(lens_before[i])):
                used.add((int(tables_before[i][t // B]), t % B))
        for blk in range(nb):
            for sl in range(B):
                if (blk, sl) not in used:
                    kp[blk, :, sl, :] = np.nan
                    vp[blk, :, sl, :] = np.inf
    return dict(
        q=torch.from_numpy(W.numpy_normal((3, q_heads, head_dim), 100)).to(dtype),
        k_pool=torch.from_numpy(kp).to(dtype), v_pool=torch.from_numpy(vp).to(dtype),
        k_new=torch.from_numpy(W.numpy_normal((3, kv_heads, head_dim), 103)).to(dtype),
        v_new=torch.from_numpy(W.numpy_normal((3, kv_heads, head_dim), 104)).to(dtype),
        slots=np.array(slots, dtype=np.int64), pairs=np.array(pairs, dtype=np.int64).reshape(-1, 2),
        lens_before=lens_before, lens_after=lens_after, tables_before=tables_before,
        tables_after=tables_after, kv_heads=kv_heads, scale=1.0 / np.sqrt(head_dim))


def random_case(seed, lens, q_heads, kv_heads, head_dim, dtype, extra_blocks=5, width=None, poison=False):
    """Sequences of the given lengths on a shuffled pool (private blocks)."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    nbs = (lens + B - 1) // B
    num_blocks = int(nbs.sum()) + extra_blocks
    perm = rng.permutation(num_blocks)
    w = width or max(1, int(nbs.max()) if len(nbs) else 1)
    tables = np.full((len(lens), w), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(nbs):
        tables[i, :n] = perm[off:off + n]
        off += n
    kp = W.numpy_normal((num_blocks, kv_heads, B, head_dim), seed * 7 + 1)
    vp = W.numpy_normal((num_blocks, kv_heads, B, head_dim), seed * 7 + 2)
    if poison:
        live = np.zeros((num_blocks, B), dtype=bool)
        for i, n in enumerate(lens):
            for t in range(int(n)):
                live[tables[i, t // B], t % B] = True
        kp.transpose(0, 2, 1, 3)[~live] = np.nan     # [blk][slot][head][d] view
        vp.transpose(0, 2, 1, 3)[~live] = -np.inf
    q = W.numpy_normal((len(lens), q_heads, head_dim), seed * 7 + 3)
    return dict(q=torch.from_numpy(q).to(dtype), k_pool=torch.from_numpy(kp).to(dtype),
                v_pool=torch.from_numpy(vp).to(dtype), tables=tables,
                lens=lens.astype(np.int32), kv_heads=kv_heads, scale=1.0 / np.sqrt(head_dim))


def attention_errors(got: torch.Tensor, want: np.ndarray):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    diff = g - want
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def grouped_case(seed, member_of, group_blocks, suffix_lens, q_heads, kv_heads, head_dim, dtype,
                 extra_blocks=3, width=None):
    """Sequences in shared-prefix groups: sequence i is in group member_of[i]
    (-1: none); the members of group p begin with the same group_blocks[p]
    blocks; sequence i then holds suffix_lens[i] tokens of its own."""
    rng = np.random.default_rng(seed)
    member_of = [int(g) for g in member_of]
    own_tokens = np.asarray(suffix_lens, dtype=np.int64)
    heads = [int(group_blocks[g]) if g >= 0 else 0 for g in member_of]
    own_blocks = (own_tokens + B - 1) // B
    num_blocks = int(sum(group_blocks)) + int(own_blocks.sum()) + extra_blocks
    perm = list(rng.permutation(num_blocks))
    shared = [[int(perm.pop()) for _ in range(nb)] for nb in group_blocks]
    lens = np.array([h * B + s for h, s in zip(heads, own_tokens)], dtype=np.int32)
    w = width or max(1, int(max(h + o for h, o in zip(heads, own_blocks))))
    tables = np.full((len(member_of), w), -1, dtype=np.int32)
    for i, g in enumerate(member_of):
        row = (shared[g] if g >= 0 else []) + [int(perm.pop()) for _ in range(int(own_blocks[i]))]
        tables[i, :len(row)] = row
    kp = W.numpy_normal((num_blocks, kv_heads, B, head_dim), seed * 11 + 1)
    vp = W.numpy_normal((num_blocks, kv_heads, B, head_dim), seed * 11 + 2)
    q = W.numpy_normal((len(member_of), q_heads, head_dim), seed * 11 + 3)
    return dict(q=torch.from_numpy(q).to(dtype), k_pool=torch.from_numpy(kp).to(dtype),
                v_pool=torch.from_numpy(vp).to(dtype), tables=tables, lens=lens,
                prefix_group=np.array(member_of, dtype=np.int32),
                group_blocks=np.array(group_blocks, dtype=np.int32), kv_heads=kv_heads,
                scale=1.0 / np.sqrt(head_dim))


def multiquery_case(seed, lens, nqs, q_heads, kv_heads, head_dim, dtype, extra_blocks=4, width=None, poison=False):
    """Sequences of the given lengths on a shuffled pool; sequence i's last
    nqs[i] tokens are its queries (rows query_start[i] .. query_start[i+1]-1).
    poison: every slot no sequence holds is K = NaN, V = -inf."""
    c = random_case(seed, lens, q_heads, kv_heads, head_dim, dtype, extra_blocks=extra_blocks, width=width,
                    poison=poison)
    qs = np.concatenate([[0], np.cumsum(np.asarray(nqs, dtype=np.int64))]).astype(np.int32)
    q = W.numpy_normal((int(qs[-1]), q_heads, head_dim), seed * 7 + 5)
    c["q"] = torch.from_numpy(q).to(dtype)
    c["query_start"] = qs
    return c
