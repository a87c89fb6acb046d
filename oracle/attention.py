"""Float64 decode attention over a paged KV cache.

Definition restated from the pages:

* Notebook 10 project demo, Demo 2 (``attention``): logits ``q k^T`` scaled
  by ``1/sqrt(d)``, the row maximum subtracted, exponentiated, normalised,
  then multiplied into ``v``. Here the scale is an explicit argument (the
  configs pass ``1/sqrt(head_dim)``).
* Notebook 10 section 3: grouped-query attention stores ``kv_heads`` K/V
  heads while the work runs over the query heads; query head ``h`` reads KV
  head ``h // (query_heads / kv_heads)`` (contiguous groups -- the plain
  reading, as the pages give no other mapping).
* Release page "NeuralOps v1.3.4", Architectural Breakdown 1 and notebook
  section 5: logical token ``t`` of sequence ``i`` lives in physical block
  ``block_tables[i][t // B]`` at slot ``t % B``.

So one output row is ``softmax(scale * K q) V`` with ``K``/``V`` the first
``context_lens[i]`` logical tokens gathered through the block table. bf16
inputs widen to float64 exactly (a bf16 value is the top 16 bits of a
float32). A sequence with no tokens has no keys to attend to; its output is
defined as zeros (notebook section 3 notes that a decode with no keys is not
a decode query that occurs in practice).

Nothing here splits the context, reorders the sum or fuses steps.
"""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return wide.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a cache or query array given as float32, bf16 bits or float64."""
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def gather_tokens(pool: np.ndarray, table, n_tokens: int, kv_head: int,
                  block_size: int = 16) -> np.ndarray:
    """Rows of logical tokens ``0..n_tokens-1`` of one KV head, in logical order.

    ``pool`` is ``[num_blocks][kv_heads][B][head_dim]``. Returns
    ``[n_tokens][head_dim]`` in the pool's own dtype.
    """
    n_blocks = -(-n_tokens // block_size)
    ids = [int(b) for b in list(table)[:n_blocks]]
    if n_blocks == 0:
        return pool[:0, kv_head, 0, :]
    rows = np.concatenate([pool[b, kv_head] for b in ids], axis=0)
    return rows[:n_tokens]


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """``softmax(scale * K q) V`` for one or more queries, all float64.

    ``q`` is ``[G][d]`` (G query heads sharing this K/V), ``K``/``V`` are
    ``[n][d]``. Returns ``[G][d]``; zeros when ``n == 0``.
    """
    q = np.atleast_2d(q)
    if K.shape[0] == 0:
        return np.zeros((q.shape[0], V.shape[1]), dtype=np.float64)
    logits = scale * (q @ K.T)                       # [G][n]
    logits = logits - logits.max(axis=1, keepdims=True)
    weights = np.exp(logits)
    weights = weights / weights.sum(axis=1, keepdims=True)
    return weights @ V                               # [G][d]


def decode_attention_pair(q, k_pool, v_pool, block_tables, context_lens, scale,
                          seq: int, kv_head: int, kv_heads: int, dtype: str,
                          block_size: int = 16) -> np.ndarray:
    """Float64 output rows of the query heads of one (sequence, KV head).

    ``q`` is ``[batch][query_heads][d]``. Returns ``[G][d]`` for query heads
    ``kv_head*G .. kv_head*G+G-1`` with ``G = query_heads // kv_heads``.
    """
    query_heads = q.shape[1]
    G = query_heads // kv_heads
    n = int(context_lens[seq])
    table = block_tables[seq]
    K = to_f64(gather_tokens(k_pool, table, n, kv_head, block_size), dtype)
    V = to_f64(gather_tokens(v_pool, table, n, kv_head, block_size), dtype)
    qg = to_f64(q[seq, kv_head * G:(kv_head + 1) * G], dtype)
    return softmax_attention(qg, K, V, scale)


def decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale,
                     kv_heads: int, dtype: str, block_size: int = 16) -> np.ndarray:
    """Float64 ``[batch][query_heads][d]`` for every sequence and query head."""
    batch, query_heads, d = q.shape
    if query_heads % kv_heads:
        raise ValueError("query_heads must be a multiple of kv_heads")
    G = query_heads // kv_heads
    out = np.zeros((batch, query_heads, d), dtype=np.float64)
    for i in range(batch):
        for j in range(kv_heads):
            out[i, j * G:(j + 1) * G] = decode_attention_pair(
                q, k_pool, v_pool, block_tables, context_lens, scale, i, j,
                kv_heads, dtype, block_size)
    return out


def contiguous_attention(q, K_seq, V_seq, scale, kv_heads: int) -> np.ndarray:
    """Unpaged reference: ``K_seq``/``V_seq`` are ``[n][kv_heads][d]`` float64
    holding the logical tokens in order, ``q`` is ``[query_heads][d]``."""
    query_heads = q.shape[0]
    G = query_heads // kv_heads
    out = np.zeros(q.shape, dtype=np.float64)
    for h in range(query_heads):
        j = h // G
        out[h] = softmax_attention(q[h:h + 1], K_seq[:, j, :], V_seq[:, j, :], scale)[0]
    return out
