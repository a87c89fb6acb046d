"""Low-bit paged KV: per-row symmetric quantization, the quantizing append and
attention over the quantized cache. Test infrastructure: only tests, the
smoke check and the bench's CPU legs use it.

Sources:

* Notebook 10, section 8 (compression): moving from 16 to fewer bits per
  coordinate shrinks the bytes per token in proportion (a storage scenario).
* Notebook 10 project demo, ``fake_quantize_rows``: per row, ``limit =
  2**(bits-1) - 1``, ``scale = max|x| / limit`` (1 when the row is zero),
  ``codes = clip(rint(x / scale), -limit, limit)``, dequantized value
  ``codes * scale``.

Reading (the notebook dequantizes in float64 and says the demo is an
experiment on the numbers, not a storage format): a row is the ``head_dim`` coordinates of one token of one
KV head. A packed cache stores the codes as int8 and the scale as a float32:
``scale = float32(max|x|) / float32(limit)`` rounded to float32 (max|x| of
bf16 or float32 inputs is exact in float32); the code decision divides in
float64 by that stored float32 scale and rounds half to even, so every code
is a function of the stored scale. The value a cached row stands for is
``code * scale`` (exact in float64). With 8 bits, ``limit = 127``.
"""

from __future__ import annotations

import numpy as np

from .attention import gather_tokens, softmax_attention, to_f64


def quantize_rows(x: np.ndarray, bits: int = 8):
    """Rows along the last axis -> (int8 codes, float32 scales with one fewer axis)."""
    if not 2 <= bits <= 8:
        raise ValueError("bits must be in [2, 8]")
    limit = 2 ** (bits - 1) - 1
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    scale = (amax / np.float32(limit)).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    codes = np.clip(np.rint(x / scale.astype(np.float64)[..., None]), -limit, limit).astype(np.int8)
    return codes, scale


def dequantize_rows(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """float64 value of a quantized row: code * scale."""
    return codes.astype(np.float64) * scale.astype(np.float64)[..., None]


def append_tokens_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, slots, block_size: int = 16):
    """Quantizing slot-mapped append (in place). ``k_new``/``v_new`` are float64
    ``[tokens][kv_heads][d]``; the code pools are ``[blocks][kv_heads][B][d]``
    int8 and the scale pools ``[blocks][kv_heads][B]`` float32. A negative slot
    skips its token."""
    kc, ks = quantize_rows(k_new)
    vc, vs = quantize_rows(v_new)
    for t, s in enumerate(np.asarray(slots).reshape(-1)):
        if s < 0:
            continue
        b, o = divmod(int(s), block_size)
        k_codes[b, :, o, :] = kc[t]
        v_codes[b, :, o, :] = vc[t]
        k_scales[b, :, o] = ks[t]
        v_scales[b, :, o] = vs[t]


def decode_attention_q8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, scale,
                        kv_heads: int, q_dtype: str, block_size: int = 16) -> np.ndarray:
    """Float64 decode attention over the values the quantized cache stands for.
    ``q`` is ``[batch][query_heads][d]`` in ``q_dtype`` ("bf16" bits or "f32")."""
    kd = dequantize_rows(k_codes, k_scales)
    vd = dequantize_rows(v_codes, v_scales)
    batch, query_heads, d = q.shape
    G = query_heads // kv_heads
    out = np.zeros((batch, query_heads, d))
    for i in range(batch):
        n = int(context_lens[i])
        for j in range(kv_heads):
            K = gather_tokens(kd, block_tables[i], n, j, block_size)
            V = gather_tokens(vd, block_tables[i], n, j, block_size)
            out[i, j * G:(j + 1) * G] = softmax_attention(to_f64(q[i, j * G:(j + 1) * G], q_dtype), K, V, scale)
    return out
