"""KV byte accounting, page-waste closed forms and attention FLOP counts.

Restates "Notebook 10. KV cache and serving: bytes, pages, and ceilings":

* section 1 ("Typed KV geometry and units"): ordinary MHA/GQA/MQA layers
  store K and V, so one token costs ``2 * layers * kv_heads * head_dim *
  bytes``; a latent-attention layer stores ``layers * (latent + rope) *
  bytes``; the payload of equal-length requests is an exact integer.
* section 3: attention work scales with the query heads while storage scales
  with the KV heads; QK and AV cost 4 FLOPs per (layer, query head, dim,
  query-key pair).
* section 6 ("Page trace and fragmentation"): naive preallocation waste and
  the expected final-block waste under a uniform remainder.

The unit policy is the notebook's: KiB/MiB/GiB are powers of two, GB/TB and
bandwidth are powers of ten.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

KIB, MIB, GIB = 2 ** 10, 2 ** 20, 2 ** 30
DECIMAL_GB = 10 ** 9


def _positive(name: str, value) -> int:
    if isinstance(value, bool) or not isinstance(value, int) or value <= 0:
        raise ValueError(f"{name} must be a positive integer")
    return value


def _non_negative(name: str, value) -> int:
    if isinstance(value, bool) or not isinstance(value, int) or value < 0:
        raise ValueError(f"{name} must be a non-negative integer")
    return value


@dataclass(frozen=True)
class KVGeometry:
    """Ordinary attention: every layer materialises K and V per KV head."""
    layers: int
    kv_heads: int
    head_dim: int
    bytes_per_element: int = 2

    def __post_init__(self):
        for name in ("layers", "kv_heads", "head_dim", "bytes_per_element"):
            _positive(name, getattr(self, name))

    @property
    def bytes_per_token(self) -> int:
        # K and V (factor 2) for every layer, KV head and head dimension.
        return 2 * self.layers * self.kv_heads * self.head_dim * self.bytes_per_element


@dataclass(frozen=True)
class LatentKVGeometry:
    """Latent attention: one stored latent plus a separate positional part."""
    layers: int
    latent_dim: int
    rope_dim: int
    bytes_per_element: int = 2

    def __post_init__(self):
        _positive("layers", self.layers)
        _positive("latent_dim", self.latent_dim)
        _non_negative("rope_dim", self.rope_dim)
        _positive("bytes_per_element", self.bytes_per_element)

    @property
    def bytes_per_token(self) -> int:
        return self.layers * (self.latent_dim + self.rope_dim) * self.bytes_per_element


def kv_payload_bytes(geometry, context_tokens: int, batch: int = 1, kv_scale: float = 1.0) -> int:
    """Exact KV bytes of ``batch`` requests of ``context_tokens`` tokens.

    ``kv_scale`` models a smaller storage format; a scaled payload that is
    not a whole number of bytes is an error, as in the notebook.
    """
    tokens = _non_negative("context_tokens", context_tokens)
    b = _positive("batch", batch)
    if isinstance(kv_scale, bool) or not math.isfinite(kv_scale) or kv_scale <= 0:
        raise ValueError("kv_scale must be positive and finite")
    raw = geometry.bytes_per_token * tokens * b * kv_scale
    whole = round(raw)
    if abs(raw - whole) > 1e-9:
        raise ValueError("scaled KV payload is not a whole number of bytes")
    return int(whole)


def naive_preallocation_waste(max_tokens: int, used_tokens: int) -> float:
    """Unused share of a fixed max-length reservation."""
    m = _positive("max_tokens", max_tokens)
    u = _non_negative("used_tokens", used_tokens)
    if u > m:
        raise ValueError("used_tokens cannot exceed max_tokens")
    return (m - u) / m


def expected_paged_waste(avg_tokens: int, block_size: int) -> float:
    """Expected unused slots over expected allocated slots.

    With a uniform remainder the last block leaves ``(B-1)/2`` slots unused
    on average, against ``avg + (B-1)/2`` allocated slots.
    """
    a = _positive("avg_tokens", avg_tokens)
    B = _positive("block_size", block_size)
    unused = (B - 1) / 2
    return unused / (a + unused)


def attention_flops(layers: int, query_heads: int, head_dim: int, queries: int,
                    cached_prefix: int = 0) -> int:
    """QK plus AV FLOPs (2 per multiply-add each) for causal suffix queries.

    Query ``j`` of the suffix sees ``cached_prefix + j + 1`` keys, so the
    number of query-key pairs is ``queries*prefix + queries*(queries+1)/2``.
    """
    for name, v in (("layers", layers), ("query_heads", query_heads), ("head_dim", head_dim),
                    ("queries", queries), ("cached_prefix", cached_prefix)):
        _non_negative(name, v)
    if min(layers, query_heads, head_dim) == 0:
        raise ValueError("attention geometry must be positive")
    pairs = queries * cached_prefix + queries * (queries + 1) // 2
    return 4 * layers * query_heads * head_dim * pairs


def decode_kv_bytes(context_lens, kv_heads: int, head_dim: int, bytes_per_element: int) -> int:
    """KV bytes one decode-attention call must read: every live token of every
    sequence, K and V, all KV heads, one layer (section 1 with one layer)."""
    return int(sum(int(n) for n in context_lens)) * 2 * kv_heads * head_dim * bytes_per_element


def decode_attention_flops(context_lens, query_heads: int, head_dim: int) -> int:
    """QK+AV FLOPs of one decode query per sequence against its whole context:
    4 FLOPs per (query head, dim, key) -- section 3's count with one layer."""
    return 4 * query_heads * head_dim * int(sum(int(n) for n in context_lens))
