"""Seeded synthetic inputs for the paged decode path (shared by tests and bench).

This module only draws random numbers and lays out index metadata. It holds
none of the attention, append or copy arithmetic, and it imports neither the
CUDA binding nor the CPU oracle, so both sides can take their inputs from it.

Workloads (named by what they are; all use 16-token blocks):

* ``tiny_f32``     -- 3 sequences, 4 query / 2 KV heads, head_dim 64, fp32,
  a 16-block pool handed out in an order drawn from seed 0.
* ``llama8k``      -- Llama-3-8B decode layer: batch 32, 32 q / 8 kv heads,
  head_dim 128, bf16, every context 8192 tokens, block tables a random
  permutation (seed 1) of a 16384-block pool.
* ``mixed``        -- continuous-batching mix: batch 256, Llama-3-8B heads,
  lengths log-uniform on [16, 32768] (seed 2), tables packed from a shuffled
  pool of exactly ``sum(ceil(len/16))`` blocks.
* ``long128k``     -- 70B GQA heads (64 q / 8 kv), batch 4, 131072 tokens
  each, tables a permutation (seed 3) of a 32768-block pool.
* ``prefix``       -- batch 64, Llama-3-8B heads, a 4096-token (256-block)
  shared prefix plus private suffixes uniform in [1, 2048] (seed 4).
* ``spec4``        -- the ``llama8k`` layer verifying 4 draft tokens per
  sequence: every context 8192 tokens including the 4 new ones, 4 causal
  queries per sequence, tables a permutation (seed 5) of a 16384-block pool.
* ``prefill512``   -- chunked prefill on the Llama-3-8B layer: batch 8,
  32 q / 8 kv heads, head_dim 128, bf16, every context 8192 tokens of which
  the last 512 are this step's chunk (512 causal queries per sequence),
  tables a permutation (seed 7) of a 4096-block pool.
* ``llama8k_q8``   -- the ``llama8k`` layer over an int8 cache: K codes
  ``[blocks][8][16][128]``, V codes ``[blocks][8][128][16]``, float32 scales
  ``[blocks][8][16]`` per pool; codes a rounded normal of standard deviation
  42 clipped to +-127, scales uniform on [0.02, 0.03] (the range per-row
  scales of standard-normal rows fall in), tables a permutation (seed 6).

Values are standard normal. Large tensors are drawn on the device with a
seeded ``torch.Generator``; the oracle reads the same tensors back, so
parity never depends on two machines drawing identical numbers.
"""

from __future__ import annotations

import math

import numpy as np

BLOCK_SIZE = 16

CONFIGS = {
    "tiny_f32": dict(batch=3, q_heads=4, kv_heads=2, head_dim=64, dtype="f32",
                     num_blocks=16, seed=0),
    "llama8k": dict(batch=32, q_heads=32, kv_heads=8, head_dim=128, dtype="bf16",
                    context=8192, num_blocks=16384, seed=1),
    "mixed": dict(batch=256, q_heads=32, kv_heads=8, head_dim=128, dtype="bf16",
                  min_len=16, max_len=32768, seed=2),
    "long128k": dict(batch=4, q_heads=64, kv_heads=8, head_dim=128, dtype="bf16",
                     context=131072, num_blocks=32768, seed=3),
    "prefix": dict(batch=64, q_heads=32, kv_heads=8, head_dim=128, dtype="bf16",
                   prefix=4096, min_suffix=1, max_suffix=2048, seed=4),
    "spec4": dict(batch=32, q_heads=32, kv_heads=8, head_dim=128, dtype="bf16",
                  context=8192, num_blocks=16384, queries=4, seed=5),
    "llama8k_q8": dict(batch=32, q_heads=32, kv_heads=8, head_dim=128, dtype="int8",
                       context=8192, num_blocks=16384, seed=6),
    "prefill512": dict(batch=8, q_heads=32, kv_heads=8, head_dim=128, dtype="bf16",
                       context=8192, num_blocks=4096, queries=512, seed=7),
}


def blocks_needed(tokens) -> np.ndarray:
    """ceil(tokens / 16) element-wise (how many blocks hold that many tokens)."""
    t = np.asarray(tokens, dtype=np.int64)
    return (t + BLOCK_SIZE - 1) // BLOCK_SIZE


def permuted_tables(num_blocks: int, batch: int, blocks_per_seq: int, seed: int) -> np.ndarray:
    """int32 [batch][blocks_per_seq]: the first batch*blocks_per_seq entries of a
    random permutation of the pool's ids (numpy ``default_rng(seed)``)."""
    perm = np.random.default_rng(seed).permutation(num_blocks)
    need = batch * blocks_per_seq
    if need > num_blocks:
        raise ValueError("pool too small")
    return perm[:need].reshape(batch, blocks_per_seq).astype(np.int32)


def log_uniform_lengths(batch: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int64 lengths ``rint(exp(U(ln lo, ln hi)))`` (numpy ``default_rng(seed)``)."""
    u = np.random.default_rng(seed).uniform(math.log(lo), math.log(hi), size=batch)
    return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int64)


def packed_tables(lengths, seed: int, extra_blocks: int = 0):
    """Tables drawing ``ceil(len/16)`` distinct ids per sequence from one shuffled
    pool of exactly ``sum(ceil(len/16)) + extra_blocks`` blocks.

    Returns ``(tables int32 [batch][max_blocks] padded with -1, num_blocks)``.
    """
    nb = blocks_needed(lengths)
    num_blocks = int(nb.sum()) + int(extra_blocks)
    perm = np.random.default_rng(seed + 1000).permutation(num_blocks)
    width = max(1, int(nb.max()))
    tables = np.full((len(nb), width), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(nb):
        tables[i, :n] = perm[off:off + n]
        off += n
    return tables, num_blocks


def uniform_suffixes(batch: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """int64 suffix lengths uniform on [lo, hi] (numpy ``default_rng(seed)``)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=batch).astype(np.int64)


def slot_of(tables: np.ndarray, positions) -> np.ndarray:
    """Physical slot id of logical position ``positions[i]`` of sequence ``i``.

    A slot id names one 16-token block row: ``block_id * 16 + offset``. This
    is how a host-side block manager addresses the new token of a step.
    """
    pos = np.asarray(positions, dtype=np.int64)
    rows = np.arange(len(pos))
    return tables[rows, pos // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + pos % BLOCK_SIZE


def numpy_normal(shape, seed: int) -> np.ndarray:
    """float32 standard normal from numpy ``default_rng(seed)`` (small inputs)."""
    return np.random.default_rng(seed).standard_normal(shape, dtype=np.float32)


def torch_normal(shape, seed: int, dtype, device):
    """Standard normal drawn by a seeded ``torch.Generator`` on ``device``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32).to(dtype)


def int8_codes(shape, seed: int, device):
    """Rounded normal draws of standard deviation 42, clipped to [-127, 127], as int8."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32) * 42.0
    return x.round().clamp_(-127, 127).to(torch.int8)


def uniform(shape, lo: float, hi: float, seed: int, device):
    """float32 draws uniform on [lo, hi)."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def workload_index(name: str):
    """Index metadata of a named workload: ``(tables int32, lens int64, num_blocks)``.

    ``lens`` are the context lengths after the step's append (the new token
    is attended to).
    """
    cfg = CONFIGS[name]
    B = cfg["batch"]
    if name in ("llama8k", "long128k", "spec4", "llama8k_q8", "prefill512"):
        lens = np.full(B, cfg["context"], dtype=np.int64)
        tables = permuted_tables(cfg["num_blocks"], B, cfg["context"] // BLOCK_SIZE, cfg["seed"])
        num_blocks = cfg["num_blocks"]
    elif name == "mixed":
        lens = log_uniform_lengths(B, cfg["min_len"], cfg["max_len"], cfg["seed"])
        tables, num_blocks = packed_tables(lens, cfg["seed"])
    elif name == "prefix":
        suffix = uniform_suffixes(B, cfg["min_suffix"], cfg["max_suffix"], cfg["seed"])
        lens = cfg["prefix"] + suffix + 1
        n_prefix = cfg["prefix"] // BLOCK_SIZE
        n_private = blocks_needed(lens) - n_prefix
        num_blocks = n_prefix + int(n_private.sum())
        perm = np.random.default_rng(cfg["seed"] + 1000).permutation(num_blocks)
        width = int(blocks_needed(lens).max())
        tables = np.full((B, width), -1, dtype=np.int32)
        off = n_prefix
        for i in range(B):
            tables[i, :n_prefix] = perm[:n_prefix]           # the shared prefix blocks
            tables[i, n_prefix:n_prefix + n_private[i]] = perm[off:off + n_private[i]]
            off += n_private[i]
    else:
        raise ValueError(f"no workload {name!r}")
    return tables.astype(np.int32), lens, num_blocks


def device_workload(name: str, device, seed_offset: int = 0) -> dict:
    """Full-size inputs of one decode step of a named workload, on ``device``.

    Returns the K/V pools, q, the step's new K/V rows with their slots, the
    copy pairs (none for these workloads), block tables and the context
    lengths *after* the step's append (the new tokens are attended to). With
    ``queries`` new tokens per sequence (``spec4``), q holds that many rows per
    sequence in sequence order and ``query_start`` gives their offsets.
    """
    import torch

    cfg = CONFIGS[name]
    bf = torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16   # int8 pools take bf16 q and new rows
    B, HQ, HKV, D = cfg["batch"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
    nq = cfg.get("queries", 1)
    seed = cfg["seed"] + seed_offset
    tables, lens, num_blocks = workload_index(name)
    # the step's new tokens: positions lens - nq .. lens - 1 of every sequence
    pos = (lens[:, None] - nq + np.arange(nq)[None, :]).reshape(-1)
    slots = slot_of(np.repeat(tables, nq, axis=0), pos)
    # shared-prefix groups: the prefix workload is one group over its shared blocks
    n_shared = cfg.get("prefix", 0) // BLOCK_SIZE
    group = np.zeros(B, dtype=np.int32) if n_shared else np.full(B, -1, dtype=np.int32)
    if cfg["dtype"] == "int8":
        # scale pool [blocks][heads][2][16]: K-row and V-row scales of a block and head together;
        # k_scales / v_scales are views of its two halves
        scales = torch.stack([uniform((num_blocks, HKV, BLOCK_SIZE), 0.02, 0.03, seed + 5, device),
                              uniform((num_blocks, HKV, BLOCK_SIZE), 0.02, 0.03, seed + 6, device)], dim=2)
        pools = dict(k_pool=int8_codes((num_blocks, HKV, BLOCK_SIZE, D), seed, device),
                     v_pool=int8_codes((num_blocks, HKV, D, BLOCK_SIZE), seed + 1, device),
                     scales=scales, k_scales=scales[:, :, 0], v_scales=scales[:, :, 1])
    else:
        pools = dict(k_pool=torch_normal((num_blocks, HKV, BLOCK_SIZE, D), seed, bf, device),
                     v_pool=torch_normal((num_blocks, HKV, BLOCK_SIZE, D), seed + 1, bf, device))
    return dict(
        name=name, cfg=cfg, num_blocks=num_blocks, **pools,
        q=torch_normal((B * nq, HQ, D), seed + 2, bf, device),
        k_new=torch_normal((B * nq, HKV, D), seed + 3, bf, device),
        v_new=torch_normal((B * nq, HKV, D), seed + 4, bf, device),
        query_start=torch.arange(0, B * nq + 1, nq, dtype=torch.int32, device=device),
        queries=nq,
        slots=torch.from_numpy(slots).to(device),
        pairs=torch.zeros((0, 2), dtype=torch.int64, device=device),
        tables=torch.from_numpy(tables).to(device),
        lens=torch.from_numpy(lens.astype(np.int32)).to(device),
        tables_np=tables, lens_np=lens.astype(np.int32), slots_np=slots,
        scale=1.0 / math.sqrt(D),
        prefix_group=torch.from_numpy(group).to(device),
        group_blocks=torch.tensor([n_shared] if n_shared else [], dtype=torch.int32, device=device),
        max_group_blocks=n_shared,
    )
