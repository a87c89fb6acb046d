"""Float64 two-phase decode attention over blocks shared by groups of
sequences. Test infrastructure: only tests, the smoke check and the bench's
CPU legs use it.

Sources:

* Paper-search page, the ChunkAttention abstract ("prefix-aware
  self-attention", KV split into chunks held in a prefix tree, "two-phase
  partition" kernel): the shared chunks are read once for all requests that
  share them.
* Notebook 10, section 5 (``share_prefix``: the target's table begins with
  the source's first ``ceil(prefix / B)`` blocks) and section 7 (prefix
  reuse): which sequences hold the same physical blocks.
* Notebook 10 project demo, Demo 2 (``attention``): the softmax attention
  whose result the two phases must reproduce.

Reading (the abstract names the phases but not their arithmetic): a *group*
is a set of sequences whose block tables begin with the same
``group_blocks[p]`` whole physical blocks. Phase 1 (chunk-first) attends the
queries of every member, all together, over the group's shared tokens and
keeps, per query head, the normalised partial output ``o`` and the natural
log-sum-exp ``lse`` of the scaled logits. Phase 2 (sequence-first) does the
same for each sequence over its remaining tokens. The two partials combine
by their ``lse`` weights::

    out = (e^(lse_1 - M) o_1 + e^(lse_2 - M) o_2) / (e^(lse_1 - M) + e^(lse_2 - M)),
    M = max(lse_1, lse_2)

which is softmax attention over the union of the two token sets. A partial
over no tokens has ``lse = -inf`` and ``o = 0``; it carries no weight.
Sequences in no group (group -1) are attended in one pass. Only whole blocks
are shared: tokens of a shared partial block belong to phase 2.
"""

from __future__ import annotations

import numpy as np

from .attention import gather_tokens, to_f64


def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Normalised partial output and natural log-sum-exp of ``scale * K q``.

    ``q`` is ``[R][d]`` (R query rows), ``K``/``V`` are ``[n][d]``, all
    float64. Returns ``(o [R][d], lse [R])``; ``(0, -inf)`` when ``n == 0``.
    """
    q = np.atleast_2d(q)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1])), np.full(q.shape[0], -np.inf)
    logits = scale * (q @ K.T)                        # [R][n]
    mx = logits.max(axis=1, keepdims=True)
    w = np.exp(logits - mx)
    s = w.sum(axis=1, keepdims=True)
    return (w / s) @ V, (mx + np.log(s))[:, 0]


def combine_partials(parts):
    """Combine ``[(o, lse), ...]`` partials of the same query rows."""
    lses = np.stack([lse for _, lse in parts])         # [P][R]
    M = lses.max(axis=0)                               # [R]
    live = np.isfinite(M)
    Msafe = np.where(live, M, 0.0)
    wts = np.where(np.isfinite(lses), np.exp(lses - Msafe), 0.0)   # [P][R]
    den = wts.sum(axis=0)
    num = sum(w[:, None] * o for w, (o, _) in zip(wts, parts))
    out = np.zeros_like(num)
    out[live] = num[live] / den[live][:, None]
    return out


def tokens_range(pool, table, first: int, last: int, kv_head: int, block_size: int = 16):
    """Rows of logical tokens ``first .. last-1`` (``first`` a multiple of the
    block size) of one KV head, in logical order."""
    if last <= first:
        return pool[:0, kv_head, 0, :]
    b0 = first // block_size
    return gather_tokens(pool, list(table)[b0:], last - first, kv_head, block_size)


def group_members(prefix_group, p: int):
    """Sequence indices of group ``p``, in index order."""
    return [i for i, g in enumerate(prefix_group) if int(g) == p]


def check_groups(block_tables, context_lens, prefix_group, group_blocks, block_size: int = 16):
    """Raise ``ValueError`` unless every member's table begins with the same
    ``group_blocks[p]`` blocks as the group's first member and its context
    holds them all."""
    for i, g in enumerate(prefix_group):
        g = int(g)
        if g < 0:
            continue
        if g >= len(group_blocks):
            raise ValueError(f"sequence {i}: group {g} out of range")
        nb = int(group_blocks[g])
        if nb < 0 or nb * block_size > int(context_lens[i]):
            raise ValueError(f"sequence {i}: {nb} shared blocks exceed its context")
        first = group_members(prefix_group, g)[0]
        if list(block_tables[i][:nb]) != list(block_tables[first][:nb]):
            raise ValueError(f"sequence {i}: table does not begin with group {g}'s blocks")


def decode_attention_two_phase(q, k_pool, v_pool, block_tables, context_lens, scale,
                               kv_heads: int, dtype: str, prefix_group, group_blocks,
                               block_size: int = 16) -> np.ndarray:
    """Float64 ``[batch][query_heads][d]`` by the two phases above."""
    check_groups(block_tables, context_lens, prefix_group, group_blocks, block_size)
    batch, query_heads, d = q.shape
    G = query_heads // kv_heads
    qf = to_f64(q, dtype)
    shared = {}                     # (sequence, kv head) -> phase-1 partial of its G rows
    for p in range(len(group_blocks)):
        members = group_members(prefix_group, p)
        if not members:
            continue
        n_shared = int(group_blocks[p]) * block_size
        table = block_tables[members[0]]
        for j in range(kv_heads):
            K = to_f64(tokens_range(k_pool, table, 0, n_shared, j, block_size), dtype)
            V = to_f64(tokens_range(v_pool, table, 0, n_shared, j, block_size), dtype)
            rows = np.concatenate([qf[i, j * G:(j + 1) * G] for i in members])   # all members at once
            o, lse = partial_attention(rows, K, V, scale)
            for r, i in enumerate(members):
                shared[(i, j)] = (o[r * G:(r + 1) * G], lse[r * G:(r + 1) * G])
    out = np.zeros((batch, query_heads, d))
    for i in range(batch):
        g = int(prefix_group[i])
        first = int(group_blocks[g]) * block_size if g >= 0 else 0
        n = int(context_lens[i])
        for j in range(kv_heads):
            K = to_f64(tokens_range(k_pool, block_tables[i], first, n, j, block_size), dtype)
            V = to_f64(tokens_range(v_pool, block_tables[i], first, n, j, block_size), dtype)
            own = partial_attention(qf[i, j * G:(j + 1) * G], K, V, scale)
            parts = [own] + ([shared[(i, j)]] if g >= 0 else [])
            out[i, j * G:(j + 1) * G] = combine_partials(parts)
    return out
