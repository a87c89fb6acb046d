"""Float64 multi-query attention over a paged KV cache. Test infrastructure:
only tests, the smoke check and the bench's CPU legs use it.

Sources:

* Release page "NeuralOps v1.3.4", Architectural Breakdown 2 (speculative
  decoding pipeline): the target model verifies the K draft tokens in one
  parallel pass.
* Notebook 10, section 7 (prefix reuse): a cached-prefix suffix "still
  attends to all cached positions", with causal query-key pairs inside the
  suffix; the chunks of a prefill together contain exactly the causal pairs
  of the whole prompt.
* Notebook 10 project demo, Demo 2 (``attention``): the softmax attention of
  one query.

Reading: sequence i holds ``context_lens[i] = n`` tokens, the last ``nq``
of which are this step's new tokens (already appended). Its queries are rows
``query_start[i] .. query_start[i+1]-1`` of ``q``; query ``t`` sits at
position ``n - nq + t`` and attends causally, to tokens ``0 .. n - nq + t``.
With one query per sequence this is the decode attention.
"""

from __future__ import annotations

import numpy as np

from .attention import gather_tokens, softmax_attention, to_f64  # noqa: F401  (softmax_attention: used by tests)


def multiquery_attention(q, k_pool, v_pool, block_tables, context_lens, query_start, scale,
                         kv_heads: int, dtype: str, block_size: int = 16) -> np.ndarray:
    """Float64 ``[total_queries][query_heads][d]``.

    Per (sequence, KV head) the queries' logits against all ``n`` gathered
    tokens are formed at once; a token a query may not see (position past
    ``n - nq + t``) gets logit ``-inf``, i.e. weight exactly 0, so each row is
    the softmax over its visible tokens only.
    """
    total, query_heads, d = q.shape
    if query_heads % kv_heads:
        raise ValueError("query_heads must be a multiple of kv_heads")
    G = query_heads // kv_heads
    out = np.zeros((total, query_heads, d))
    for i in range(len(context_lens)):
        q0, q1 = int(query_start[i]), int(query_start[i + 1])
        n, nq = int(context_lens[i]), q1 - q0
        if nq > n:
            raise ValueError(f"sequence {i}: {nq} queries but {n} tokens")
        if nq == 0:
            continue
        last_visible = n - nq + np.arange(nq)                       # query t sees tokens 0 .. last_visible[t]
        visible = np.arange(n)[None, :] <= last_visible[:, None]   # [nq][n]
        visible = np.repeat(visible, G, axis=0)                    # rows (t, g)
        for j in range(kv_heads):
            K = to_f64(gather_tokens(k_pool, block_tables[i], n, j, block_size), dtype)
            V = to_f64(gather_tokens(v_pool, block_tables[i], n, j, block_size), dtype)
            Q = to_f64(q[q0:q1, j * G:(j + 1) * G], dtype).reshape(nq * G, d)
            logits = np.where(visible, scale * (Q @ K.T), -np.inf)
            logits = logits - logits.max(axis=1, keepdims=True)
            weights = np.exp(logits)
            weights = weights / weights.sum(axis=1, keepdims=True)
            out[q0:q1, j * G:(j + 1) * G] = (weights @ V).reshape(nq, G, d)
    return out
