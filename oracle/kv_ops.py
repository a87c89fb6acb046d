"""Block copy and slot-mapped append on host arrays (exact byte moves).

The cache layout is ``pool[num_blocks][kv_heads][B][head_dim]`` with K and V
in separate pools, ``B`` = 16 tokens per physical block ("NeuralOps v1.3.4"
release page, Architectural Breakdown 1: fixed 16-token physical blocks, a
block table from logical tokens to physical blocks, slot mapping for
concurrent requests). A slot id is ``block * B + offset``; a negative slot
means "no write" (a padded token).

Copy-on-write ("Notebook 10 ...", section 5): before a sequence appends into a
shared partial final block, the block is duplicated into a private block.
The copy moves the whole block -- every KV head and every slot -- for K and V.

Both functions work on any dtype (bf16 arrives as uint16 bit patterns) and
move bytes only, so the result is exact by construction.
"""

from __future__ import annotations

import numpy as np


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs) -> None:
    """Copy block ``src`` onto block ``dst`` for every ``(src, dst)``, in place.

    All sources are read before any destination is written, i.e. the copies
    act as one simultaneous step. (A valid copy list has distinct
    destinations that are not also sources, for which this equals doing the
    pairs one after another.)
    """
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    if len(pairs) == 0:
        return
    for pool in (k_pool, v_pool):
        staged = pool[pairs[:, 0]].copy()
        pool[pairs[:, 1]] = staged


def append_tokens(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray,
                  v_new: np.ndarray, slot_mapping, block_size: int = 16) -> None:
    """Write token ``t``'s K/V rows (all heads) into slot ``slot_mapping[t]``.

    ``k_new``/``v_new`` are ``[T][kv_heads][head_dim]``. Slot ``s`` addresses
    ``pool[s // B, :, s % B, :]``; negative slots are skipped.
    """
    slots = np.asarray(slot_mapping, dtype=np.int64).reshape(-1)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        block, offset = divmod(int(s), block_size)
        k_pool[block, :, offset, :] = k_new[t]
        v_pool[block, :, offset, :] = v_new[t]
