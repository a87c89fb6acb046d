"""Checks that tie the float64 attention oracle and the byte-move oracle to
something other than themselves. Each pin raises ``AssertionError`` on failure.

They are plain functions (not collected as tests) so that
``test_oracle_attention.py`` can run them against the oracle and
``test_oracle_mutants.py`` can run them against planted mistakes, showing
that a plausible error (a dropped term, a wrong index, a transposed operand)
fails at least one of them.

What each pin compares with:

* ``pin_sdpa``            -- PyTorch's own ``scaled_dot_product_attention``
  in float64 over the *contiguous* logical K/V, with the grouped heads
  expanded by ``repeat_interleave`` (the notebook's "PyTorch bridge - B17"
  check: attention over the cache equals attention over the full keys).
* ``pin_single_token``    -- one key: softmax weight exactly 1, output = v0.
* ``pin_constant_keys``   -- equal logits: output = mean of V.
* ``pin_dominant_key``    -- a logit 1000 above the rest: output = that key's
  V (also shows the maximum is subtracted: exp(1000) overflows).
* ``pin_scale_zero``      -- scale 0: output = mean of V.
* ``pin_permutation``     -- relabelling physical blocks changes nothing.
* ``pin_garbage_outside`` -- NaN/inf in slots past the context and in
  unreferenced blocks never reach the output.
* ``pin_append`` / ``pin_copy`` -- exactly the addressed rows / blocks
  change, byte for byte.
* ``pin_append_then_gather`` -- tokens appended through their slots are
  read back in logical order.
"""

from __future__ import annotations

import numpy as np

import oracle.attention as A
import oracle.kv_ops as K

B = 16


def _place(pool, tables, seq_tokens):
    """Write logical token t of sequence i (all heads) into block
    tables[i][t // B], slot t % B. Plain loops; independent of the oracle."""
    for i, toks in enumerate(seq_tokens):
        for t in range(toks.shape[0]):
            pool[tables[i][t // B], :, t % B, :] = toks[t]


def _problem(seed, lens, kv_heads=2, q_heads=4, d=8, extra_blocks=3):
    rng = np.random.default_rng(seed)
    nb = [(n + B - 1) // B for n in lens]
    num_blocks = sum(nb) + extra_blocks
    ids = rng.permutation(num_blocks)
    width = max(nb + [1])
    tables = np.full((len(lens), width), -1, dtype=np.int64)
    off = 0
    for i, n in enumerate(nb):
        tables[i, :n] = ids[off:off + n]
        off += n
    ks = [rng.standard_normal((n, kv_heads, d)) for n in lens]
    vs = [rng.standard_normal((n, kv_heads, d)) for n in lens]
    kp = rng.standard_normal((num_blocks, kv_heads, B, d))
    vp = rng.standard_normal((num_blocks, kv_heads, B, d))
    _place(kp, tables, ks)
    _place(vp, tables, vs)
    q = rng.standard_normal((len(lens), q_heads, d))
    return dict(q=q, kp=kp.astype(np.float32), vp=vp.astype(np.float32), tables=tables,
                lens=np.array(lens), ks=ks, vs=vs, kv_heads=kv_heads, d=d)


def _oracle(p, scale, q=None):
    return A.decode_attention((p["q"] if q is None else q).astype(np.float32), p["kp"], p["vp"],
                              p["tables"], p["lens"], scale, p["kv_heads"], "f32")


def pin_sdpa():
    import torch
    import torch.nn.functional as F
    for seed, lens in ((1, [5, 19, 33]), (2, [1, 16, 17, 48])):
        p = _problem(seed, lens)
        scale = 0.37
        got = _oracle(p, scale)
        G = p["q"].shape[1] // p["kv_heads"]
        for i, n in enumerate(lens):
            k = torch.tensor(p["ks"][i].astype(np.float32).astype(np.float64)).permute(1, 0, 2)
            v = torch.tensor(p["vs"][i].astype(np.float32).astype(np.float64)).permute(1, 0, 2)
            k = k.repeat_interleave(G, dim=0)
            v = v.repeat_interleave(G, dim=0)
            q = torch.tensor(p["q"][i].astype(np.float32).astype(np.float64)).unsqueeze(1)
            want = F.scaled_dot_product_attention(q, k, v, scale=scale).squeeze(1).numpy()
            assert np.allclose(got[i], want, rtol=0, atol=1e-12), (seed, i)


def pin_single_token():
    p = _problem(3, [1, 1], extra_blocks=0)
    got = _oracle(p, 0.5)
    G = 2
    for i in range(2):
        for h in range(4):
            assert np.array_equal(got[i, h], p["vs"][i][0, h // G].astype(np.float32).astype(np.float64))


def pin_constant_keys():
    p = _problem(4, [7, 40])
    for i, n in enumerate([7, 40]):
        p["ks"][i][:] = p["ks"][i][0]
    _place(p["kp"], p["tables"], p["ks"])
    got = _oracle(p, 0.9)
    for i, n in enumerate([7, 40]):
        for h in range(4):
            want = p["vs"][i][:, h // 2].astype(np.float32).astype(np.float64).mean(axis=0)
            assert np.allclose(got[i, h], want, rtol=0, atol=1e-13)


def pin_dominant_key():
    p = _problem(5, [30], d=4, kv_heads=1, q_heads=1)
    q = np.zeros((1, 1, 4))
    q[0, 0, 0] = 1.0
    p["ks"][0][:] = 0.0
    p["ks"][0][17, 0, 0] = 1000.0
    _place(p["kp"], p["tables"], p["ks"])
    got = _oracle(p, 1.0, q=q)
    want = p["vs"][0][17, 0].astype(np.float32).astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.allclose(got[0, 0], want, rtol=0, atol=1e-15)


def pin_scale_zero():
    p = _problem(6, [9, 21])
    got = _oracle(p, 0.0)
    for i in range(2):
        for h in range(4):
            want = p["vs"][i][:, h // 2].astype(np.float32).astype(np.float64).mean(axis=0)
            assert np.allclose(got[i, h], want, rtol=0, atol=1e-13)


def pin_permutation():
    p = _problem(7, [3, 18, 35])
    base = _oracle(p, 0.3)
    nbk = p["kp"].shape[0]
    perm = np.random.default_rng(70).permutation(nbk)      # old id -> new id
    kp2 = np.empty_like(p["kp"])
    vp2 = np.empty_like(p["vp"])
    kp2[perm] = p["kp"]
    vp2[perm] = p["vp"]
    t2 = np.where(p["tables"] >= 0, perm[np.maximum(p["tables"], 0)], -1)
    got = A.decode_attention(p["q"].astype(np.float32), kp2, vp2, t2, p["lens"], 0.3, 2, "f32")
    assert np.array_equal(got, base)


def pin_garbage_outside():
    p = _problem(8, [5, 20])
    base = _oracle(p, 0.4)
    used = set()
    for i, n in enumerate([5, 20]):
        for t in range(n):
            used.add((int(p["tables"][i][t // B]), t % B))
    for blk in range(p["kp"].shape[0]):
        for s in range(B):
            if (blk, s) not in used:
                p["kp"][blk, :, s, :] = np.nan
                p["vp"][blk, :, s, :] = np.inf
    got = _oracle(p, 0.4)
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, base)


def pin_append():
    rng = np.random.default_rng(9)
    kp = rng.standard_normal((6, 2, B, 4)).astype(np.float32)
    vp = rng.standard_normal((6, 2, B, 4)).astype(np.float32)
    k0, v0 = kp.copy(), vp.copy()
    kn = np.ones((3, 2, 4), np.float32) * np.array([1, 2, 3], np.float32)[:, None, None]
    vn = -kn
    kn[:, 1] += 10
    slots = [4 * B + 3, -1, 0 * B + 15]
    K.append_tokens(kp, vp, kn, vn, slots)
    changed = np.argwhere(np.any(kp != k0, axis=3))
    assert sorted(map(tuple, changed)) == [(0, 0, 15), (0, 1, 15), (4, 0, 3), (4, 1, 3)]
    assert np.array_equal(kp[4, :, 3], kn[0]) and np.array_equal(vp[4, :, 3], vn[0])
    assert np.array_equal(kp[0, :, 15], kn[2]) and np.array_equal(vp[0, :, 15], vn[2])
    assert np.array_equal(np.argwhere(np.any(vp != v0, axis=3)), changed)


def pin_copy():
    rng = np.random.default_rng(10)
    kp = rng.standard_normal((8, 2, B, 4)).astype(np.float32)
    vp = rng.standard_normal((8, 2, B, 4)).astype(np.float32)
    k0, v0 = kp.copy(), vp.copy()
    K.copy_blocks(kp, vp, [(1, 6), (3, 0)])
    assert np.array_equal(kp[6], k0[1]) and np.array_equal(kp[0], k0[3])
    assert np.array_equal(vp[6], v0[1]) and np.array_equal(vp[0], v0[3])
    for b in (1, 2, 3, 4, 5, 7):
        assert np.array_equal(kp[b], k0[b]) and np.array_equal(vp[b], v0[b])
    K.copy_blocks(kp, vp, np.zeros((0, 2), np.int64))
    assert np.array_equal(kp[6], k0[1])


def pin_append_then_gather():
    rng = np.random.default_rng(11)
    kp = np.full((5, 2, B, 4), np.nan, np.float32)
    vp = np.full((5, 2, B, 4), np.nan, np.float32)
    table = [3, 0, 4]
    toks_k = rng.standard_normal((40, 2, 4)).astype(np.float32)
    toks_v = rng.standard_normal((40, 2, 4)).astype(np.float32)
    slots = [table[t // B] * B + t % B for t in range(40)]
    K.append_tokens(kp, vp, toks_k, toks_v, slots)
    for h in range(2):
        assert np.array_equal(A.gather_tokens(kp, table, 40, h), toks_k[:, h])
        assert np.array_equal(A.gather_tokens(vp, table, 33, h), toks_v[:33, h])


def pin_bf16_widening():
    """bf16 bits widen exactly: checked against torch's own bf16 -> float64."""
    import torch
    x = torch.randn(4096, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(A.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())
    special = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F80, 0x0001], np.uint16)
    w = A.bf16_bits_to_f64(special)
    assert w[0] == 0.0 and w[2] == 1.0 and w[3] == -1.0 and np.isinf(w[4]) and w[5] == 2.0 ** -133


ALL_PINS = [pin_sdpa, pin_single_token, pin_constant_keys, pin_dominant_key, pin_scale_zero,
            pin_permutation, pin_garbage_outside, pin_append, pin_copy, pin_append_then_gather,
            pin_bf16_widening]
